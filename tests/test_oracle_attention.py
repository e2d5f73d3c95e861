"""Pins of the fp64 decode-attention oracle against facts fixed by the mathematics
of scaled dot-product attention and by an independent library routine (the
page "Perplexity libera o Lily", section "O modelo em tres formatos de carga":
grouped-query attention, 16 query heads over two KV heads; section "Prefill e
decode": a fixed-block KV cache)."""
import numpy as np
import pytest
import torch

import oracle
from bit_grouped_expert_top_gb300.attn_inputs import ATTN_CONFIGS, make_attn


def bf16_bits(a) -> np.ndarray:
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(rng, B=2, H_q=16, H_kv=2, D=64, bs=16, lens=(5, 40), extra=2):
    nb = [(L + bs - 1) // bs for L in lens]
    n_blocks = sum(nb) + extra
    q = bf16_bits(rng.standard_normal((B, H_q, D)))
    k = bf16_bits(rng.standard_normal((n_blocks, H_kv, bs, D)))
    v = bf16_bits(rng.standard_normal((n_blocks, H_kv, bs, D)))
    perm = rng.permutation(n_blocks).astype(np.int32)
    table = np.full((B, max(nb)), -1, np.int32)
    at = 0
    for b, n in enumerate(nb):
        table[b, :n] = perm[at:at + n]
        at += n
    return q, k, v, table, np.array(lens, np.int32)


def _gather(cache, table, L, g, bs):
    """Rows of kv head g of one sequence, in token order (values as float64)."""
    rows = [cache[table[t // bs], g, t % bs] for t in range(L)]
    return bf16_value(np.stack(rows))


def test_single_token_returns_its_value_row():
    # softmax over one score is 1: every head returns the value row of its group
    rng = np.random.default_rng(1)
    q, k, v, table, lens = _case(rng, lens=(1, 1))
    out = oracle.attn_decode(q, k, v, table, lens)
    for b in range(2):
        for h in range(16):
            np.testing.assert_array_equal(out[b, h], bf16_value(v[table[b, 0], h // 8, 0]))


def test_equal_keys_average_the_values():
    # all keys of a head equal: uniform weights, the output is the mean value row
    rng = np.random.default_rng(2)
    q, k, v, table, lens = _case(rng, lens=(23, 48))
    k[:] = k[0, 0, 0]
    out = oracle.attn_decode(q, k, v, table, lens)
    for b, L in enumerate(lens):
        for g in range(2):
            mean = _gather(v, table[b], L, g, 16).mean(axis=0)
            for h in range(8 * g, 8 * g + 8):
                np.testing.assert_allclose(out[b, h], mean, rtol=0, atol=1e-12)


def test_matches_torch_scaled_dot_product_attention():
    # an independent library routine (PyTorch's CPU attention in float64) on the
    # gathered cache rows, with the KV heads repeated over their query groups
    rng = np.random.default_rng(3)
    q, k, v, table, lens = _case(rng, D=32, lens=(17, 64))
    out = oracle.attn_decode(q, k, v, table, lens)
    for b, L in enumerate(lens):
        K = np.stack([_gather(k, table[b], L, g, 16) for g in range(2)])  # [H_kv][L][D]
        V = np.stack([_gather(v, table[b], L, g, 16) for g in range(2)])
        Kq = torch.from_numpy(np.repeat(K, 8, axis=0))[:, None]          # [H_q][1][L][D]
        Vq = torch.from_numpy(np.repeat(V, 8, axis=0))[:, None]
        Q = torch.from_numpy(bf16_value(q[b]))[:, None, None]             # [H_q][1][1][D]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kq, Vq)[:, 0, 0].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_explicit_scale_is_applied():
    # scale s on (q, k) equals the default 1/sqrt(D) on (q * s * sqrt(D), k):
    # scaling q by 2 (exact in bf16) with scale/2 gives the same scores
    rng = np.random.default_rng(4)
    q, k, v, table, lens = _case(rng, lens=(9, 33))
    q2 = bf16_bits(bf16_value(q) * 2.0)
    a = oracle.attn_decode(q, k, v, table, lens, scale=0.3)
    b = oracle.attn_decode(q2, k, v, table, lens, scale=0.15)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_block_placement_does_not_matter():
    # moving each logical block to another physical block (and the table with it)
    # leaves the result unchanged, bit for bit
    rng = np.random.default_rng(5)
    q, k, v, table, lens = _case(rng, lens=(30, 61), extra=4)
    out = oracle.attn_decode(q, k, v, table, lens)
    n = k.shape[0]
    perm = rng.permutation(n)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v
    t2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(oracle.attn_decode(q, k2, v2, t2, lens), out)


def test_query_heads_read_only_their_kv_head():
    # heads 0..7 read KV head 0 only: changing KV head 1 changes heads 8..15 alone
    rng = np.random.default_rng(6)
    q, k, v, table, lens = _case(rng, lens=(12, 50))
    out = oracle.attn_decode(q, k, v, table, lens)
    k2, v2 = k.copy(), v.copy()
    k2[:, 1] = bf16_bits(rng.standard_normal(k2[:, 1].shape))
    v2[:, 1] = bf16_bits(rng.standard_normal(v2[:, 1].shape))
    out2 = oracle.attn_decode(q, k2, v2, table, lens)
    np.testing.assert_array_equal(out2[:, :8], out[:, :8])
    assert np.abs(out2[:, 8:] - out[:, 8:]).min() > 0


def test_dominant_key_selects_its_value():
    # one key far more aligned with q than the rest: its weight tends to 1
    rng = np.random.default_rng(7)
    q, k, v, table, lens = _case(rng, B=1, H_q=1, H_kv=1, lens=(40,))
    qv = bf16_value(q[0, 0])
    t = 29
    blk, row = table[0, t // 16], t % 16
    k[blk, 0, row] = bf16_bits(qv * 8.0)           # score 8 |q|^2 / sqrt(D), far above the others
    out = oracle.attn_decode(q, k, v, table, lens)
    np.testing.assert_allclose(out[0, 0], bf16_value(v[blk, 0, row]), rtol=0, atol=1e-9)


def test_generated_workload_is_consistent():
    # the tiny workload: every used block exists and the tables cover the lengths
    cfg = ATTN_CONFIGS["attn_tiny"]
    a = make_attn(cfg)
    assert a["q"].shape == (cfg.B, cfg.H_q, cfg.D)
    n_blocks = a["k_cache"].shape[0]
    for b, L in enumerate(cfg.seq_lens):
        used = a["block_table"][b, : (L + cfg.block_size - 1) // cfg.block_size]
        assert bool((used >= 0).all()) and bool((used < n_blocks).all())
    out = oracle.attn_decode(*(a[n].view(torch.int16).numpy().view(np.uint16) if a[n].dtype == torch.bfloat16
                               else a[n].numpy() for n in ("q", "k_cache", "v_cache", "block_table", "seq_lens")))
    assert np.isfinite(out).all()
