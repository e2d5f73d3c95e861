"""GPU parity of grouped-query decode attention over a fixed-block KV cache
(lily_attn_decode) against the fp64 oracle.

Tolerance, from the arithmetic: the scores are fp32 sums of exact bf16
products (their error moves a weight by ~1e-6 relative), and the softmax
weights are rounded to bf16 before they multiply V, with the normaliser summed
over the rounded weights.  A weight is then off by at most 2^-9 relative and
its normalised value by at most 2^-8, so per output element
    |o_gpu - o| <= 2^-8 * sum_t w_t |v_t| + 1e-5,
and sum_t w_t |v_t| is the oracle run with |V| in place of V.
"""
import numpy as np
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
import oracle
from bit_grouped_expert_top_gb300.attn_inputs import ATTN_CONFIGS, AttnConfig, make_attn

pytestmark = pytest.mark.gpu

INDEX_ERR = -7  # LILY_ERR_DEVICE_INDEX


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _run(a, cfg, scale=None):
    dev = {k: v.cuda() for k, v in a.items()}
    s = lm.make_attn_shape(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.block_size, a["block_table"].shape[1])
    ws = lm.alloc_attn_workspace(s)
    out = torch.full((cfg.B, cfg.H_q, cfg.D), float("nan"), dtype=torch.float32, device="cuda")
    lm.lily_attn_decode(s, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seq_lens"], out, ws,
                        scale=scale)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), lm.lily_moe_device_status(ws), (s, dev, ws, out)


def _oracle(a, scale=None, abs_v=False):
    v = _bits(a["v_cache"])
    if abs_v:
        v = v & np.uint16(0x7FFF)
    return oracle.attn_decode(_bits(a["q"]), _bits(a["k_cache"]), v, a["block_table"].numpy(),
                              a["seq_lens"].numpy(), scale)


def _check(a, cfg, scale=None):
    got, st, _ = _run(a, cfg, scale)
    assert st == 0, lm.lily_moe_status_string(st)
    ref = _oracle(a, scale)
    bound = 2.0 ** -8 * _oracle(a, scale, abs_v=True) + 1e-5
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= bound).all(), f"max err {err.max():.3e}, worst ratio {(err / bound).max():.3f}"
    return got


def test_tiny_three_sequences():
    # lengths 1, 100 (ragged last block) and 777 over a shuffled cache
    cfg = ATTN_CONFIGS["attn_tiny"]
    _check(make_attn(cfg), cfg)


@pytest.mark.parametrize("D,bs", [(64, 32), (64, 128), (128, 32), (128, 128), (256, 32), (256, 64)])
def test_head_dims_and_block_sizes(D, bs):
    cfg = AttnConfig("sweep", seq_lens=(bs, 3 * bs + 5, 1000), D=D, block_size=bs, seed=20 + D + bs)
    _check(make_attn(cfg), cfg)


@pytest.mark.parametrize("H_q,H_kv", [(16, 2), (8, 2), (4, 4), (2, 1), (6, 3)])
def test_group_sizes(H_q, H_kv):
    # GQA groups of 8, 4, 1, 2 and 2 query heads per KV head
    cfg = AttnConfig("groups", seq_lens=(257, 64), H_q=H_q, H_kv=H_kv, D=128, seed=30 + H_q)
    _check(make_attn(cfg), cfg)


def test_explicit_scale():
    cfg = ATTN_CONFIGS["attn_tiny"]
    _check(make_attn(cfg), cfg, scale=0.2)


def test_empty_sequence_gives_zeros():
    cfg = AttnConfig("empty", seq_lens=(0, 70), D=64, seed=40)
    a = make_attn(cfg)
    got, st, _ = _run(a, cfg)
    assert st == 0
    assert (got[0] == 0).all()
    ref = _oracle({**a, "seq_lens": a["seq_lens"][1:], "q": a["q"][1:], "block_table": a["block_table"][1:]})
    assert np.abs(got[1] - ref[0]).max() < 2e-2


def test_many_sequences_more_ctas_than_splits():
    # a decode batch of 24 sequences of mixed lengths: few splits per sequence
    lens = tuple(int(x) for x in np.random.default_rng(5).integers(1, 3000, 24))
    cfg = AttnConfig("batch", seq_lens=lens, D=128, seed=41)
    _check(make_attn(cfg), cfg)


def test_one_split_per_group():
    # 160 sequences x 2 KV heads: more groups than the GPU holds CTAs, so each
    # group is one CTA that normalises its own result (no barrier); lengths
    # 0 .. 400 tokens, one block to seven blocks
    lens = tuple(int(x) for x in np.random.default_rng(6).integers(0, 400, 160))
    cfg = AttnConfig("wide", seq_lens=lens, D=128, block_size=64, seed=43)
    _check(make_attn(cfg), cfg)


def test_many_calls_on_one_workspace():
    # the barrier words are reset by every call: twenty calls on one workspace,
    # all bit-identical, no status recorded
    cfg = AttnConfig("reuse", seq_lens=(5000,), D=256, block_size=64, seed=44)
    got, st, (s, dev, ws, out) = _run(make_attn(cfg), cfg)
    assert st == 0
    first = out.clone()
    for _ in range(20):
        out.fill_(float("nan"))
        lm.lily_attn_decode(s, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seq_lens"], out, ws)
    torch.cuda.synchronize()
    assert torch.equal(first, out)
    assert lm.lily_moe_device_status(ws) == 0


@pytest.mark.parametrize("name", ["attn_32k", "attn_128k"])
def test_full_size_contexts(name):
    # the benchmark's workloads, in its launch configuration (every head checked)
    cfg = ATTN_CONFIGS[name]
    _check(make_attn(cfg), cfg)


def test_repeat_call_is_bit_identical():
    cfg = ATTN_CONFIGS["attn_tiny"]
    got, st, (s, dev, ws, out) = _run(make_attn(cfg), cfg)
    first = out.clone()
    out.zero_()
    lm.lily_attn_decode(s, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"], dev["seq_lens"], out, ws)
    torch.cuda.synchronize()
    assert torch.equal(first, out)


def test_bad_table_entry_and_length_are_reported():
    cfg = AttnConfig("bad", seq_lens=(100, 50), D=64, seed=42)
    a = make_attn(cfg)
    a["block_table"][0, 1] = a["k_cache"].shape[0] + 7    # past the cache
    _, st, _ = _run(a, cfg)
    assert st == INDEX_ERR
    a = make_attn(cfg)
    a["seq_lens"][1] = a["block_table"].shape[1] * cfg.block_size + 1   # longer than the table
    _, st, _ = _run(a, cfg)
    assert st == INDEX_ERR


def test_host_checks():
    s = lm.make_attn_shape(1, 16, 2, 96, 64, 4)     # D outside {64, 128, 256}
    assert lm.lily_attn_workspace_bytes(s) == 0
    s = lm.make_attn_shape(1, 16, 2, 256, 128, 4)   # block too large for two ring stages
    assert lm.lily_attn_workspace_bytes(s) == 0
    s = lm.make_attn_shape(1, 18, 2, 128, 64, 4)    # 9 query heads per KV head
    assert lm.lily_attn_workspace_bytes(s) == 0


def test_shared_memory_sizes_in_any_order():
    # launches that need more, then less, then more shared memory in one process
    # (the kernel's shared-memory limit must only ever be raised)
    for D, bs in ((64, 128), (64, 32), (64, 128), (256, 64), (64, 32), (256, 64)):
        cfg = AttnConfig("order", seq_lens=(3 * bs + 1,), D=D, block_size=bs, seed=50 + D + bs)
        _check(make_attn(cfg), cfg)
