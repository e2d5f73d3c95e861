"""GPU parity of the Gated DeltaNet scan (lily_gdn_scan) against the fp64 oracle.

Tolerance, from the arithmetic: every step rounds the fp32 state update and
the two length-d_k dot products (about (d_k + 4) 2^-24 relative to the state's
size per step); the recurrence map alpha (I - beta k k^T) has norm <= 1 for
beta in [0, 1] and unit k, so old errors do not grow, and with alpha in
[0.9, 1] they fade over about 1 / (1 - mean alpha) = 20 steps.  That puts
the error near 1e-4 of the output's rms; the tests allow 1e-3.
"""
import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
import oracle
from bit_grouped_expert_top_gb300.gdn_inputs import GDN_CONFIGS, GDNConfig, make_gdn

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _gpu(g, state=True, scale=None):
    d = {k: v.cuda() for k, v in g.items()}
    T, H_v, d_v = d["v"].shape
    d_k = d["k"].shape[2]
    out = torch.full((T, H_v, d_v), float("nan"), device="cuda")
    st = torch.full((H_v, d_v, d_k), float("nan"), device="cuda")
    lm.lily_gdn_scan(d["q"], d["k"], d["v"], d["alpha"], d["beta"], out, st,
                     state_in=d.get("state") if state else None, scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), st.cpu().numpy().astype(np.float64)


def _oracle(g, state=True, scale=None):
    d_k = g["k"].shape[2]
    S0 = g["state"].numpy().astype(np.float64) if (state and "state" in g) else None
    return oracle.gdn_scan(_bits(g["q"]), _bits(g["k"]), _bits(g["v"]), g["alpha"].numpy(), g["beta"].numpy(), S0,
                           scale=1.0 / np.sqrt(d_k) if scale is None else scale)


def _check(g, state=True, scale=None):
    o, S = _gpu(g, state, scale)
    ro, rS = _oracle(g, state, scale)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    eo = np.abs(o - ro).max() / max(np.sqrt((ro ** 2).mean()), 1e-30)
    es = np.abs(S - rS).max() / max(np.sqrt((rS ** 2).mean()), 1e-30)
    assert eo <= TOL and es <= TOL, (eo, es)
    return o, S


@pytest.mark.parametrize("state", [True, False])
def test_tiny(state):
    _check(make_gdn(GDN_CONFIGS["gdn_tiny"]), state)


@pytest.mark.parametrize("T,H_k,H_v,d_k,d_v", [(300, 2, 4, 128, 128), (65, 1, 1, 128, 32), (129, 2, 8, 64, 256),
                                               (1, 4, 4, 128, 64), (200, 3, 6, 64, 48), (40, 1, 16, 128, 1024),
                                               (33, 2, 2, 64, 16)])
def test_shapes(T, H_k, H_v, d_k, d_v):
    # ragged chunks (300 = 4 x 64 + 44), one token (a decode step), group sizes 1, 2, 4
    # and 16, one to sixty-four 16-row slices per head (d_v from 16 to the largest, 1024)
    cfg = GDNConfig("shape", T=T, H_k=H_k, H_v=H_v, d_k=d_k, d_v=d_v, seed=T + d_v)
    _check(make_gdn(cfg))


def test_explicit_scale():
    _check(make_gdn(GDN_CONFIGS["gdn_tiny"]), scale=0.3)


def test_zero_tokens_copies_the_state():
    g = make_gdn(GDNConfig("t0", T=0, H_k=2, H_v=4, d_k=64, d_v=32, seed=3))
    _, S = _gpu(g)
    assert np.array_equal(S, g["state"].numpy().astype(np.float64))


def test_two_calls_continue_one_scan_exactly():
    # the state out of the first part is the state in of the second: the same
    # fp32 operations in the same order, so the results are bit-identical
    g = make_gdn(GDNConfig("cont", T=200, H_k=2, H_v=4, d_k=128, d_v=64, seed=4))
    o, S = _gpu(g)
    first = {k: (v[:120].contiguous() if k != "state" else v) for k, v in g.items()}
    o1, S1 = _gpu(first)
    second = {k: (v[120:].contiguous() if k != "state" else torch.from_numpy(S1.astype(np.float32)))
              for k, v in g.items()}
    o2, S2 = _gpu(second)
    assert np.array_equal(np.concatenate([o1, o2]), o)
    assert np.array_equal(S2, S)


@pytest.mark.parametrize("T,d_k", [(31, 128), (32, 128), (33, 64), (64, 128), (96, 64), (97, 128)])
def test_chunk_pipeline_edges(T, d_k):
    # whole and ragged 32-token chunks at the ends of the staging pipeline
    # (one, two and three chunks; the last chunk full or one token long)
    cfg = GDNConfig("edge", T=T, H_k=2, H_v=4, d_k=d_k, d_v=32, seed=T + d_k)
    _check(make_gdn(cfg))


@pytest.mark.parametrize("split", [1, 37, 64, 95])
def test_split_anywhere_continues_exactly(split):
    # a scan split at any token (inside a chunk, on a chunk boundary, one token
    # in) repeats the single call's bits
    g = make_gdn(GDNConfig("split", T=130, H_k=2, H_v=4, d_k=128, d_v=32, seed=7))
    o, S = _gpu(g)
    first = {k: (v[:split].contiguous() if k != "state" else v) for k, v in g.items()}
    o1, S1 = _gpu(first)
    second = {k: (v[split:].contiguous() if k != "state" else torch.from_numpy(S1.astype(np.float32)))
              for k, v in g.items()}
    o2, S2 = _gpu(second)
    assert np.array_equal(np.concatenate([o1, o2]), o)
    assert np.array_equal(S2, S)


def test_small_and_zero_decay():
    # alpha of 1e-6, and 0 on every seventh token (the state is then replaced by
    # the token's own write): still within the bound of the oracle
    g = make_gdn(GDNConfig("smalla", T=100, H_k=2, H_v=4, d_k=64, d_v=32, seed=5))
    g["alpha"] = torch.full_like(g["alpha"], 1e-6)
    g["alpha"][::7] = 0.0
    _check(g)


def test_repeat_is_bit_identical():
    g = make_gdn(GDN_CONFIGS["gdn_t512"])
    a = _gpu(g)
    b = _gpu(g)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name", ["gdn_t512", "gdn_t8192"])
def test_full_size(name):
    # the benchmark's workloads (16 key heads, 32 value heads of 128), every output
    _check(make_gdn(GDN_CONFIGS[name]))


def test_host_checks():
    g = {k: v.cuda() for k, v in make_gdn(GDN_CONFIGS["gdn_tiny"]).items()}
    out = torch.empty_like(g["v"], dtype=torch.float32)
    st = torch.empty_like(g["state"])
    with pytest.raises(lm.LilyError):  # state_out aliasing state_in
        lm.lily_gdn_scan(g["q"], g["k"], g["v"], g["alpha"], g["beta"], out, g["state"], state_in=g["state"])
    bad = torch.zeros((37, 2, 96), dtype=torch.bfloat16, device="cuda")  # d_k = 96
    with pytest.raises(lm.LilyError):
        lm.lily_gdn_scan(bad, bad, g["v"], g["alpha"], g["beta"], out, st)
