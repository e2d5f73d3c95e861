"""GPU parity of the prefill path (lily_moe_forward through the C ABI) against
the fp64 oracle: routing tables bit-exact, logits and layer outputs within the
stated bounds.  Full oracle comparison on small and ragged shapes; sampled
tokens on the full-size workloads (the same configs the benchmark runs)."""
import numpy as np
import pytest
import torch

from bit_grouped_expert_top_gb300.inputs import CONFIGS, LayerConfig
import bit_grouped_expert_top_gb300 as lm
from gpu_util import (Layer, assert_logits_close, assert_out_close, assert_routing_exact, oracle_layer_out,
                      run_forward, shape_of, x_for)
from helpers import bits

pytestmark = pytest.mark.gpu

TINY = CONFIGS["tiny"]


def _full_check(cfg: LayerConfig, T: int, block_rows=None, overrides=None, seed_offset=0, poison=False):
    layer = Layer(cfg, overrides=overrides)
    x = x_for(cfg, T=T, seed_offset=seed_offset)
    res = run_forward(cfg, layer, x, block_rows=block_rows, poison_workspace=poison)
    xb = bits(x)
    assert_logits_close(cfg, layer, xb, res["logits"])
    assert_routing_exact(cfg, res, block_rows=block_rows)
    ref = oracle_layer_out(cfg, layer, xb, res["logits"])
    return assert_out_close(res["out"], ref), res


def test_tiny_config_full_parity():
    err, res = _full_check(TINY, TINY.T)
    assert err < 1e-2


@pytest.mark.parametrize("T", [1, 3, 17, 127, 300])
def test_ragged_token_counts(T):
    _full_check(TINY, T, seed_offset=T)


@pytest.mark.parametrize("T", [512, 513, 1000, 1025, 2048, 2049])
def test_routing_chunk_regimes(T):
    # the routing runs in one launch up to 64 chunks, with 8-token chunks up to
    # T = 512, 16-token chunks up to 1024 and 32-token chunks up to 2048, and as
    # three launches above: the edges of each regime, full parity
    _full_check(TINY, T, seed_offset=T)


@pytest.mark.parametrize("block_rows", [16, 32, 64])
def test_block_rows_variants(block_rows):
    _full_check(TINY, 200, block_rows=block_rows, seed_offset=block_rows)


def test_all_tokens_forced_to_eight_experts():
    # +100 logit bias on 8 experts: every token picks exactly these; 248 experts get 0 rows,
    # each chosen expert gets T rows (several full blocks and a ragged tail).
    bias = torch.zeros(256, dtype=torch.float32)
    chosen = [3, 40, 41, 100, 128, 200, 254, 255]
    bias[chosen] = 100.0
    err, res = _full_check(TINY, 300, overrides={"router_bias": bias})
    counts = res["counts"]
    assert (counts[chosen] == 300).all() and counts.sum() == 300 * 8
    assert res["n_blocks"] == 8 * 3


def test_zero_routed_weights_leave_shared_expert():
    cfg = TINY
    L = Layer(cfg)
    over = {}
    for n in ("gate", "up", "down"):
        over[n + "_q"] = torch.zeros_like(L.t[n + "_q"])
        over[n + "_b"] = torch.zeros_like(L.t[n + "_b"])
    _full_check(cfg, 64, overrides=over)


@pytest.mark.parametrize("I", [256, 384, 1024])
def test_intermediate_sizes(I):
    # K of the down projection is I: 4, 8 and 16 k-steps (384 pads 6 k-steps to 8
    # and has a group count that is not a multiple of 8).
    cfg = TINY.with_(I=I, I_shared=I)
    _full_check(cfg, 100, seed_offset=I)


def test_route_then_experts_in_separate_calls():
    # routing tables from lily_moe_route, then lily_moe_grouped_gemm with a workspace
    # of its own: the expert path derives the inverse permutation from perm itself
    cfg, T = TINY, 150
    layer = Layer(cfg)
    x = x_for(cfg, T=T, seed_offset=11)
    s = shape_of(cfg, T)
    rt = lm.alloc_routing(s)
    lm.lily_moe_route(s, layer.w, x, lm.make_routing(rt), lm.alloc_workspace(s))
    ws2 = lm.alloc_workspace(s)
    out = torch.full((T, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
    lm.lily_moe_grouped_gemm(s, layer.w, x, lm.make_routing(rt), out, ws2)
    torch.cuda.synchronize()
    assert lm.lily_moe_device_status(ws2) == 0
    ref = oracle_layer_out(cfg, layer, bits(x), rt["logits"].cpu().numpy())
    assert_out_close(out.cpu().numpy(), ref)


def test_medium_full_hidden_size():
    # d = 2048, I = 512 at a token count the oracle finishes in seconds:
    # many weight tiles per unit and ragged expert groups.
    cfg = CONFIGS["prefill_t512"].with_(T=48)
    _full_check(cfg, 48)


def block_spread_tokens(res, T: int, block_rows: int, per_shared_block: int = 2, seed: int = 0):
    """Tokens that touch every block of the launch: one token of every routed
    block-map entry (a random row of the entry) and per_shared_block tokens of
    every block_rows-token range (the shared expert's blocks), plus the first
    and last token."""
    rng = np.random.default_rng(seed)
    toks = {0, T - 1}
    for e, p0, rows in res["block_map"]:
        toks.add(int(res["perm"][p0 + rng.integers(rows)]) // 8)
    for b0 in range(0, T, block_rows):
        n = min(block_rows, T - b0)
        toks.update(int(t) for t in b0 + rng.choice(n, size=min(per_shared_block, n), replace=False))
    return np.array(sorted(toks), dtype=np.int64)


@pytest.mark.parametrize("name", ["prefill_t512", "prefill_t2048_zipf"])
def test_full_size_workloads_every_token(name):
    # the whole output of the 512-token and the Zipf-skewed 2048-token workloads
    cfg = CONFIGS[name]
    layer = Layer(cfg)
    x = x_for(cfg)
    res = run_forward(cfg, layer, x)
    xb = bits(x)
    assert_logits_close(cfg, layer, xb, res["logits"])
    assert_routing_exact(cfg, res)
    assert_out_close(res["out"], oracle_layer_out(cfg, layer, xb, res["logits"]))
    if cfg.zipf_s is not None:
        counts = res["counts"]
        assert (counts == 0).sum() >= 1 and (counts > 300).sum() >= 2


def test_full_size_t8192_tokens_of_every_block():
    cfg = CONFIGS["prefill_t8192"]
    layer = Layer(cfg)
    x = x_for(cfg)
    res = run_forward(cfg, layer, x)
    xb = bits(x)
    assert_routing_exact(cfg, res)
    toks = block_spread_tokens(res, cfg.T, cfg.block_rows, seed=cfg.seed)
    assert len(toks) >= 128
    # every routed block and every shared block has a sampled token
    sampled = np.zeros(cfg.T, bool)
    sampled[toks] = True
    for e, p0, rows in res["block_map"]:
        assert sampled[res["perm"][p0:p0 + rows] // 8].any()
    assert_logits_close(cfg, layer, xb, res["logits"], toks)
    assert_out_close(res["out"][toks], oracle_layer_out(cfg, layer, xb, res["logits"], toks))


def test_poisoned_workspace_and_output_guards():
    # the workspace starts as all-ones bytes (NaN / -1): nothing may rely on it
    # being zero; every output buffer has a guard tail (checked in run_forward)
    _full_check(TINY, 300, seed_offset=5, poison=True)
    _full_check(CONFIGS["prefill_t512"].with_(T=48), 48, seed_offset=6, poison=True)


def test_repeat_calls_are_deterministic():
    # Routing is bit-reproducible.  The layer output is not: the down projection
    # adds each token's nine weighted expert rows into out with fp32 atomic adds,
    # whose order varies from run to run, so out may differ in its last bits
    # (a few fp32 ulps of the nine-term sum).
    cfg = TINY
    layer = Layer(cfg)
    x = x_for(cfg, T=100)
    a = run_forward(cfg, layer, x)
    b = run_forward(cfg, layer, x)
    for k in ("topk_idx", "counts", "offsets", "perm", "block_map"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["logits"], b["logits"])
    np.testing.assert_array_equal(a["topk_w"], b["topk_w"])
    scale = np.abs(a["out"]).max()
    assert np.max(np.abs(a["out"] - b["out"])) <= 8 * np.finfo(np.float32).eps * scale
