"""The allocation-free routing entry point (lily_moe_route_noalloc).

Some callers may not allocate device memory when they run the layer (a plugin
living inside another engine's fixed memory budget, or a serving loop that
forbids allocation after start-up), so they cannot hand lily_moe_route its
workspace.  lily_moe_route_noalloc keeps that scratch in a fixed device array
inside the library instead.  This file checks, through the C ABI, that two
calls in a row give the same routing as lily_moe_route on the same inputs.
It is collected last on purpose (file name), and must pass alone too.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x
from gpu_util import LOGIT_TOL, shape_of

KEYS = ("topk_idx", "counts", "offsets", "perm", "block_map", "n_blocks")


def test_noalloc_rejects_sizes_above_its_scratch_without_gpu():
    s = lm.make_shape(T=8193, d=2048)
    w = lm._abi.lily_moe_weights()
    r = lm._abi.lily_moe_routing()
    rc = lm.load().lily_moe_route_noalloc(ctypes.byref(s), ctypes.byref(w), None, ctypes.byref(r), None, None)
    assert rc in (-1, -8)  # null pointers are reported first when present
    fake = 0x10000000
    for n, _ in r._fields_:
        setattr(r, n, fake)
    w.router_w = fake
    for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(w, n, lm._abi.lily_q4(fake, fake, fake))
    rc = lm.load().lily_moe_route_noalloc(ctypes.byref(s), ctypes.byref(w), fake, ctypes.byref(r), None, None)
    assert rc == -8 and "scratch" in lm.lily_moe_status_string(rc)


def _route_pair(cfg, T, seed_offset):
    layer = make_layer(cfg, "cuda")
    w = lm.make_weights(layer)
    x = make_x(cfg, "cuda", seed_offset=seed_offset, T=T)
    s = shape_of(cfg, T)
    ref_t = lm.alloc_routing(s)
    ws = lm.alloc_workspace(s)
    lm.lily_moe_route(s, w, x, lm.make_routing(ref_t), ws)
    assert lm.lily_moe_device_status(ws) == 0
    return layer, w, x, s, ref_t


@pytest.mark.gpu
def test_noalloc_matches_workspace_route_on_two_calls_in_a_row():
    # the largest T the fixed scratch is sized for, a Zipf-routed case and a small one
    cases = [(CONFIGS["prefill_t8192"], 8192, 3), (CONFIGS["prefill_t2048_zipf"], 2048, 1), (CONFIGS["tiny"], 300, 2)]
    prepared = [_route_pair(cfg, T, so) for cfg, T, so in cases]
    torch.cuda.synchronize()
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for (cfg, T, _), (layer, w, x, s, ref_t) in zip(cases, prepared):
        got_t = lm.alloc_routing(s)
        for v in got_t.values():
            v.fill_(-1)
        lm.lily_moe_route_noalloc(s, w, x, lm.make_routing(got_t), device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        nb = int(ref_t["n_blocks"].item())
        for k in KEYS:
            a, b = got_t[k].cpu().numpy(), ref_t[k].cpu().numpy()
            if k == "block_map":
                a, b = a[:nb], b[:nb]
            np.testing.assert_array_equal(a, b, err_msg=k)
        np.testing.assert_allclose(got_t["topk_w"].cpu().numpy(), ref_t["topk_w"].cpu().numpy(), rtol=0, atol=2e-6)
        lg_ref = ref_t["logits"].cpu().numpy()
        assert np.max(np.abs(got_t["logits"].cpu().numpy() - lg_ref)) <= LOGIT_TOL * max(1.0, float(np.sqrt(np.mean(lg_ref ** 2))))


@pytest.mark.gpu
def test_noalloc_t0_writes_ok_status():
    # no tokens: nothing runs, but the call's status (OK) still reaches device_status
    cfg = CONFIGS["tiny"]
    layer = make_layer(cfg, "cuda")  # the weight tensors must outlive the call
    w = lm.make_weights(layer)
    s = shape_of(cfg, 0)
    rt = lm.alloc_routing(lm.make_shape(T=1, d=cfg.d, I=cfg.I))
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    lm.lily_moe_route_noalloc(s, w, None, lm.make_routing(rt), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_noalloc_status_is_cleared_between_calls():
    # The scratch keeps the last call's contents, its status word included.  A
    # call whose bounded wait runs out (test-only library variant: the router
    # GEMM stalls for T == 77) leaves LILY_ERR_DEVICE_TIMEOUT there; the next
    # call must start from a cleared status and report OK.  The variant is a
    # separate library with its own scratch array, built from the same code.
    from bit_grouped_expert_top_gb300 import _abi
    from bit_grouped_expert_top_gb300.build import STALL_TEST_T
    L = _abi.load_variant("stalltest")
    cfg = CONFIGS["tiny"]
    layer = make_layer(cfg, "cuda")  # the weight tensors must outlive the calls
    w = lm.make_weights(layer)
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for T, want in ((STALL_TEST_T, -6), (STALL_TEST_T + 23, 0), (STALL_TEST_T, -6), (STALL_TEST_T + 23, 0)):
        x = make_x(cfg, "cuda", seed_offset=T, T=T)
        s = shape_of(cfg, T)
        got_t = lm.alloc_routing(s)
        rc = L.lily_moe_route_noalloc(ctypes.byref(s), ctypes.byref(w), x.data_ptr(),
                                      ctypes.byref(lm.make_routing(got_t)), status.data_ptr(), stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert int(status.item()) == want, (T, int(status.item()))
        if want == 0:
            ref_t = lm.alloc_routing(s)
            lm.lily_moe_route(s, w, x, lm.make_routing(ref_t), lm.alloc_workspace(s))
            torch.cuda.synchronize()
            for k in ("topk_idx", "counts", "offsets", "perm"):
                np.testing.assert_array_equal(got_t[k].cpu().numpy(), ref_t[k].cpu().numpy(), err_msg=k)
