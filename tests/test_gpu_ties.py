"""GPU parity of the top-8 tie rule: among equal logits the lower expert index
wins, and the kept slots are ordered by descending logit, lower index first.

The router scores 256 experts and keeps eight (page "Perplexity libera o Lily",
section "O modelo em tres formatos de carga"); the tie rule and the softmax
renormalisation over the eight are the workload's routing contract.  Random
logits almost never tie, so these cases plant ties on purpose and run them
through both selection sites: the prefill routing kernels (lily_moe_route /
lily_moe_forward) and the decode kernels (lily_moe_decode, trace).

Ties are planted by giving whole classes of experts identical router rows and
biases: every member of a class then gets bitwise the same logit, whatever the
token.  Class sizes 1..22 with members spread over the expert indices put ties
inside one lane's eight experts and across lanes, and a per-token random input
decides which classes rank first, so the top-8 boundary splits a class on most
tokens (checked below: the test fails if it did not).
"""
import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
import oracle
from bit_grouped_expert_top_gb300.inputs import CONFIGS
from gpu_util import Layer, assert_out_close, assert_routing_exact, oracle_layer_out, run_forward, shape_of, x_for
from helpers import bits

pytestmark = pytest.mark.gpu

TINY = CONFIGS["tiny"]


def class_router(cfg, seed=5):
    """Router rows and biases shared by classes of experts (sizes 1, 2, ..., 22
    over a seeded permutation of the experts; the last 3 experts form a class
    of their own).  Returns (router_w bf16 [E, d], router_bias f32 [E], class id [E])."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(cfg.E)
    cls = np.empty(cfg.E, np.int64)
    pos, c = 0, 0
    while pos < cfg.E:
        n = min(c + 1, cfg.E - pos)
        cls[order[pos:pos + n]] = c
        pos += n
        c += 1
    g = torch.Generator().manual_seed(seed)
    rows = (torch.randn((c, cfg.d), generator=g) / np.sqrt(cfg.d)).to(torch.bfloat16)
    biases = (torch.randn((c,), generator=g) * 0.5).to(torch.float32)
    cls_t = torch.from_numpy(cls)
    return rows[cls_t].contiguous(), biases[cls_t].contiguous(), cls


def boundary_ties(lg: np.ndarray, idx: np.ndarray) -> int:
    """Tokens whose 8th kept logit equals the logit of an expert left out."""
    n = 0
    for t in range(lg.shape[0]):
        kept = np.zeros(lg.shape[1], bool)
        kept[idx[t]] = True
        if np.any(lg[t, ~kept] == lg[t, idx[t, -1]]):
            n += 1
    return n


def test_zero_router_selects_experts_0_to_7_with_equal_weights():
    # every logit is exactly 0: the eight lowest indices, each weight exactly 1/8
    L = Layer(TINY, overrides={"router_w": torch.zeros((TINY.E, TINY.d), dtype=torch.bfloat16)})
    x = x_for(TINY, T=70, seed_offset=21)
    res = run_forward(TINY, L, x)
    assert np.all(res["logits"] == 0.0)
    np.testing.assert_array_equal(res["topk_idx"], np.tile(np.arange(8, dtype=np.int32), (70, 1)))
    assert np.all(res["topk_w"] == np.float32(0.125))
    assert_routing_exact(TINY, res)
    assert_out_close(res["out"], oracle_layer_out(TINY, L, bits(x), res["logits"]))


def test_signed_zero_logits_tie():
    # zero router, all-negative inputs (every product is -0) and a bias of -0.0 on
    # experts 0..127: where the sum of the -0 products stays -0, experts 0..127
    # get the logit -0 and experts 128..255 the logit +0.  The two are equal,
    # so experts 0..7 win with 1/8 each; a selection that ranked -0 below +0
    # would pick experts 128..135 instead.
    bias = torch.zeros(TINY.E, dtype=torch.float32)
    bias[:128] = -0.0
    L = Layer(TINY, overrides={"router_w": torch.zeros((TINY.E, TINY.d), dtype=torch.bfloat16),
                               "router_bias": bias})
    x = -x_for(TINY, T=40, seed_offset=22).abs() - 0.25
    res = run_forward(TINY, L, x)
    assert np.all(res["logits"] == 0.0)
    np.testing.assert_array_equal(res["topk_idx"], np.tile(np.arange(8, dtype=np.int32), (40, 1)))
    assert np.all(res["topk_w"] == np.float32(0.125))
    assert_routing_exact(TINY, res)


@pytest.mark.parametrize("T", [97, 300])
def test_prefill_class_ties_match_oracle(T):
    rw, rb, _ = class_router(TINY)
    L = Layer(TINY, overrides={"router_w": rw, "router_bias": rb})
    x = x_for(TINY, T=T, seed_offset=30 + T)
    res = run_forward(TINY, L, x)
    assert_routing_exact(TINY, res)  # selection bit-exact with the oracle on the same logits
    assert boundary_ties(res["logits"], res["topk_idx"]) >= T // 2
    assert_out_close(res["out"], oracle_layer_out(TINY, L, bits(x), res["logits"]))


def test_prefill_class_ties_full_hidden_size():
    cfg = CONFIGS["prefill_t512"].with_(T=64)
    rw, rb, _ = class_router(cfg, seed=6)
    L = Layer(cfg, overrides={"router_w": rw, "router_bias": rb})
    x = x_for(cfg, T=64, seed_offset=7)
    res = run_forward(cfg, L, x)
    assert_routing_exact(cfg, res)
    assert boundary_ties(res["logits"], res["topk_idx"]) >= 32


@pytest.mark.parametrize("T", [1, 4, 8])
def test_decode_class_ties_match_oracle(T):
    cfg = TINY
    n_layers = 3
    rw, rb, _ = class_router(cfg, seed=8)
    layers = [Layer(cfg, layer_index=l, overrides={"router_w": rw, "router_bias": rb}) for l in range(n_layers)]
    s = shape_of(cfg, T)
    ws = lm.alloc_workspace(s, n_layers_decode=n_layers)
    x = x_for(cfg, T=T, seed_offset=40 + T)
    out = torch.empty((n_layers, T, cfg.d), dtype=torch.float32, device="cuda")
    x_next = torch.empty((n_layers, T, cfg.d), dtype=torch.bfloat16, device="cuda")
    trace = {"logits": torch.empty((n_layers, T, cfg.E), dtype=torch.float32, device="cuda"),
             "topk_idx": torch.empty((n_layers, T, cfg.top_k), dtype=torch.int32, device="cuda"),
             "topk_w": torch.empty((n_layers, T, cfg.top_k), dtype=torch.float32, device="cuda")}
    lm.lily_moe_decode(s, [L.w for L in layers], x, out, ws, x_next=x_next, trace=trace)
    assert lm.lily_moe_device_status(ws) == 0
    lg = trace["logits"].cpu().numpy()
    tidx = trace["topk_idx"].cpu().numpy()
    tw = trace["topk_w"].cpu().numpy()
    xn = bits(x_next)
    out_np = out.cpu().numpy()
    n_ties = 0
    for l in range(n_layers):
        idx, w = oracle.select(lg[l].astype(np.float64), cfg.top_k)
        np.testing.assert_array_equal(tidx[l], idx)
        np.testing.assert_allclose(tw[l], w, atol=2e-6, rtol=0)
        n_ties += boundary_ties(lg[l], tidx[l])
        x_l = bits(x) if l == 0 else xn[l - 1]
        ref = oracle.moe_tokens(layers[l].np, x_l, idx, w, d=cfg.d, E=cfg.E, I=cfg.I, I_shared=cfg.I_shared)
        assert_out_close(out_np[l], ref)
    assert n_ties >= 1


def test_decode_zero_router_selects_experts_0_to_7():
    cfg, T = TINY, 2
    L = Layer(cfg, overrides={"router_w": torch.zeros((cfg.E, cfg.d), dtype=torch.bfloat16)})
    s = shape_of(cfg, T)
    ws = lm.alloc_workspace(s, n_layers_decode=1)
    x = x_for(cfg, T=T, seed_offset=50)
    out = torch.empty((1, T, cfg.d), dtype=torch.float32, device="cuda")
    trace = {"topk_idx": torch.empty((1, T, 8), dtype=torch.int32, device="cuda"),
             "topk_w": torch.empty((1, T, 8), dtype=torch.float32, device="cuda")}
    lm.lily_moe_decode(s, [L.w], x, out, ws, trace=trace)
    assert lm.lily_moe_device_status(ws) == 0
    np.testing.assert_array_equal(trace["topk_idx"].cpu().numpy()[0], np.tile(np.arange(8, dtype=np.int32), (T, 1)))
    assert np.all(trace["topk_w"].cpu().numpy() == np.float32(0.125))
