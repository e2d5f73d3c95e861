"""GPU parity of the decode path (lily_moe_decode, 1..8 tokens, layers chained
by the parameter-free RMS norm) against the fp64 oracle, teacher-forced per
layer: layer l of the oracle runs on the GPU's own bf16 input of layer l."""
import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
import oracle
from bit_grouped_expert_top_gb300.inputs import CONFIGS
from gpu_util import Layer, assert_out_close, logit_error_bound, shape_of, x_for
from helpers import bits
from oracle import numpy_ref as npr

pytestmark = pytest.mark.gpu


def _run_decode(cfg, n_layers, T):
    layers = [Layer(cfg, layer_index=l) for l in range(n_layers)]
    s = shape_of(cfg, T)
    ws = lm.alloc_workspace(s, n_layers_decode=n_layers)
    x = x_for(cfg, T=T, seed_offset=100 + T)
    out = torch.empty((n_layers, T, cfg.d), dtype=torch.float32, device="cuda")
    x_next = torch.empty((n_layers, T, cfg.d), dtype=torch.bfloat16, device="cuda")
    trace = {"logits": torch.empty((n_layers, T, cfg.E), dtype=torch.float32, device="cuda"),
             "topk_idx": torch.empty((n_layers, T, cfg.top_k), dtype=torch.int32, device="cuda"),
             "topk_w": torch.empty((n_layers, T, cfg.top_k), dtype=torch.float32, device="cuda")}
    lm.lily_moe_decode(s, [L.w for L in layers], x, out, ws, x_next=x_next, trace=trace)
    assert lm.lily_moe_device_status(ws) == 0
    torch.cuda.synchronize()
    return layers, x, out, x_next, trace, ws, s


def _check_decode(cfg, n_layers, T):
    layers, x, out, x_next, trace, _, _ = _run_decode(cfg, n_layers, T)
    out_np = out.cpu().numpy()
    xn = bits(x_next)
    lg = trace["logits"].cpu().numpy()
    tidx = trace["topk_idx"].cpu().numpy()
    tw = trace["topk_w"].cpu().numpy()
    for l, L in enumerate(layers):
        x_l = bits(x) if l == 0 else xn[l - 1]
        ref_lg = oracle.logits(x_l, L.np["router_w"], L.np.get("router_bias"))
        bound = logit_error_bound(x_l, L.np["router_w"], L.np.get("router_bias"))
        assert np.all(np.abs(lg[l].astype(np.float64) - ref_lg) <= bound)
        idx, w = oracle.select(lg[l].astype(np.float64), cfg.top_k)
        np.testing.assert_array_equal(tidx[l], idx)
        np.testing.assert_allclose(tw[l], w, atol=2e-6, rtol=0)
        ref = oracle.moe_tokens(L.np, x_l, idx, w, d=cfg.d, E=cfg.E, I=cfg.I, I_shared=cfg.I_shared)
        assert_out_close(out_np[l], ref)
        # the exported next input is the RMS norm of this layer's GPU output, rounded to bf16
        want = oracle.rms_norm(out_np[l].astype(np.float64))
        got = npr.bf16_to_f64(xn[l])
        assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-3)) <= 2.0 ** -8


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_tiny_chain(T):
    _check_decode(CONFIGS["tiny"], n_layers=3, T=T)


@pytest.mark.parametrize("T", [1, 8])
def test_decode_full_size_layers(T):
    cfg = CONFIGS["decode_t1_l40"]
    _check_decode(cfg, n_layers=2, T=T)


def test_decode_repeat_call_is_bit_identical():
    cfg = CONFIGS["tiny"]
    layers, x, out, x_next, trace, ws, s = _run_decode(cfg, 2, 4)
    first = out.clone()
    first_x = x_next.clone()
    out.zero_()
    lm.lily_moe_decode(s, [L.w for L in layers], x, out, ws, x_next=x_next, trace=trace)
    torch.cuda.synchronize()
    assert torch.equal(first, out) and torch.equal(first_x, x_next)


def test_decode_more_layers_than_one_launch():
    # a long chain: every layer's input is the normalised output of the one before
    cfg = CONFIGS["tiny"]
    _check_decode(cfg, n_layers=45, T=1)


def test_decode_matches_prefill_on_same_tokens():
    cfg = CONFIGS["tiny"]
    T = 4
    layers, x, out, _, _, _, _ = _run_decode(cfg, 1, T)
    s = shape_of(cfg, T)
    ws = lm.alloc_workspace(s)
    out_p = torch.empty((T, cfg.d), dtype=torch.float32, device="cuda")
    lm.lily_moe_forward(s, layers[0].w, x, out_p, ws)
    torch.cuda.synchronize()
    ref = out_p.cpu().numpy().astype(np.float64)
    assert_out_close(out[0].cpu().numpy(), ref)
