"""The fp16 range of the expert GEMM operands is detected on the device.

The expert GEMMs multiply fp16 operands (the rebuilt 4-bit weights, x and the
SwiGLU product h) with fp32 accumulation.  A finite bf16 x, or an fp32 h, at
or beyond 65520 in magnitude would round to infinity on conversion; the
kernels record LILY_ERR_DEVICE_RANGE in the status word instead of leaving a
silent inf.  Both conversion sites are checked, in prefill and in decode; after
clearing the status the same workspace serves a normal call.
"""
import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
from bit_grouped_expert_top_gb300.inputs import CONFIGS
from gpu_util import Layer, assert_out_close, oracle_layer_out, run_forward, shape_of, x_for
from helpers import bits

pytestmark = pytest.mark.gpu

TINY = CONFIGS["tiny"]
RANGE = -9  # LILY_ERR_DEVICE_RANGE


def _forward_status(cfg, layer, x):
    s = shape_of(cfg, x.shape[0])
    ws = lm.alloc_workspace(s)
    out = torch.empty((x.shape[0], cfg.d), dtype=torch.float32, device="cuda")
    lm.lily_moe_forward(s, layer.w, x, out, ws)
    return lm.lily_moe_device_status(ws), ws


def _decode_status(cfg, layer, x):
    s = shape_of(cfg, x.shape[0])
    ws = lm.alloc_workspace(s, n_layers_decode=1)
    out = torch.empty((1, x.shape[0], cfg.d), dtype=torch.float32, device="cuda")
    lm.lily_moe_decode(s, [layer.w], x, out, ws)
    return lm.lily_moe_device_status(ws)


def _x_overflow(T, seed_offset):
    # a few entries of 1e5 (bf16 99840): finite in bf16, infinite in fp16
    x = x_for(TINY, T=T, seed_offset=seed_offset)
    x[T // 2, 7] = 1e5
    x[0, TINY.d - 1] = -1e5
    return x


def _x_h_overflow(T, seed_offset):
    # |x| ~ 300 fits fp16, but gate and up reach a few hundred, so silu(g) * u
    # passes 65504 for many elements
    return (x_for(TINY, T=T, seed_offset=seed_offset).float() * 300.0).to(torch.bfloat16)


def test_prefill_flags_x_beyond_fp16():
    L = Layer(TINY)
    st, ws = _forward_status(TINY, L, _x_overflow(64, 1))
    assert st == RANGE, lm.lily_moe_status_string(st)
    # the status is sticky until cleared; then the same workspace runs a normal call
    assert lm.lily_moe_device_status(ws) == RANGE
    lm.lily_moe_clear_status(ws)
    s = shape_of(TINY, 64)
    x = x_for(TINY, T=64, seed_offset=2)
    rt = lm.alloc_routing(s)
    out = torch.empty((64, TINY.d), dtype=torch.float32, device="cuda")
    lm.lily_moe_forward(s, L.w, x, out, ws, routing=lm.make_routing(rt))
    assert lm.lily_moe_device_status(ws) == 0
    ref = oracle_layer_out(TINY, L, bits(x), rt["logits"].cpu().numpy())
    assert_out_close(out.cpu().numpy(), ref)


def test_prefill_flags_h_beyond_fp16():
    L = Layer(TINY)
    x = _x_h_overflow(64, 3)
    assert float(x.float().abs().max()) < 65504
    st, _ = _forward_status(TINY, L, x)
    assert st == RANGE, lm.lily_moe_status_string(st)


def test_prefill_in_range_large_inputs_pass():
    # |x| up to a few hundred with h well inside fp16 (x scaled by 20): no flag
    L = Layer(TINY)
    x = (x_for(TINY, T=64, seed_offset=4).float() * 20.0).to(torch.bfloat16)
    res = run_forward(TINY, L, x)  # asserts status 0
    assert_out_close(res["out"], oracle_layer_out(TINY, L, bits(x), res["logits"]))


def test_decode_flags_x_beyond_fp16():
    assert _decode_status(TINY, Layer(TINY), _x_overflow(2, 5)) == RANGE


def test_decode_flags_h_beyond_fp16():
    assert _decode_status(TINY, Layer(TINY), _x_h_overflow(1, 6)) == RANGE
