"""Failure detection on the GPU without a GPU fault.

Every pipeline wait of the grouped GEMM is bounded: when one runs out the
kernel records LILY_ERR_DEVICE_TIMEOUT in the workspace status word, every role
gives up, the copies and tensor-core work already in flight drain, tensor
memory is freed and the kernel returns, so the CUDA context stays usable.

The product library never waits long enough for that to happen, so these
tests load the test-only build variant (liblily_moe_stalltest.so: pipeline
waits limited to 1 ms, and for T == 77 the epilogue first waits on a barrier
that nothing completes).  The waits on the exit path keep their full 2 s
limit in that variant.  After the timeout the same process runs a normal call
through the product library and checks it against the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
from bit_grouped_expert_top_gb300 import _abi
from bit_grouped_expert_top_gb300.build import STALL_TEST_T
from bit_grouped_expert_top_gb300.inputs import CONFIGS
from gpu_util import Layer, assert_out_close, assert_routing_exact, oracle_layer_out, run_forward, shape_of, x_for
from helpers import bits

pytestmark = pytest.mark.gpu

TINY = CONFIGS["tiny"]
TIMEOUT = -6  # LILY_ERR_DEVICE_TIMEOUT


def _stall_forward(layer, x):
    L = _abi.load_variant("stalltest")
    T = x.shape[0]
    s = shape_of(TINY, T)
    ws = lm.alloc_workspace(s)
    out = torch.zeros((T, TINY.d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.lily_moe_forward(ctypes.byref(s), ctypes.byref(layer.w), x.data_ptr(), out.data_ptr(), None,
                            ws.data_ptr(), ws.numel(), stream)
    assert rc == 0
    return L.lily_moe_device_status(ws.data_ptr(), stream), out


def test_bounded_wait_times_out_then_the_gpu_runs_a_normal_call():
    layer = Layer(TINY)
    x = x_for(TINY, T=STALL_TEST_T, seed_offset=9)
    st, _ = _stall_forward(layer, x)
    assert st == TIMEOUT, lm.lily_moe_status_string(st)
    torch.cuda.synchronize()
    # the context is intact: the product library computes the same layer correctly
    res = run_forward(TINY, layer, x)
    assert_routing_exact(TINY, res)
    assert_out_close(res["out"], oracle_layer_out(TINY, layer, bits(x), res["logits"]))


def test_stall_variant_is_the_product_path_for_other_sizes():
    # with T != 77 the test variant computes the layer like the product library
    layer = Layer(TINY)
    x = x_for(TINY, T=STALL_TEST_T + 1, seed_offset=10)
    st, out = _stall_forward(layer, x)
    assert st == 0
    res = run_forward(TINY, layer, x)
    assert_out_close(out.cpu().numpy(), oracle_layer_out(TINY, layer, bits(x), res["logits"]))
