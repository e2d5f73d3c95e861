"""Pins of the fp64 CPU oracle against things other than itself.

Each test pins one part of the oracle with a closed form, a hand-derived value,
an invariant, a special case, brute force, or an independent vectorised
formulation using library primitives (numpy matmul / stable sort / bincount).
The method is the one on the page "Perplexity libera o Lily" (noticiai.com.br):
section "O modelo em tres formatos de carga" (256 experts, top-8, one shared
expert) and section "Prefill e decode" (4-bit group-64 affine weights with bf16
scale and bias; histogram, prefix scan, scatter and block map of the routing).
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import numpy_ref as npr
from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x
from helpers import bits, rel_max_err, small_cfg, small_layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(v: float) -> int:
    """Bits of an exactly representable bf16 value (test-side helper)."""
    b = np.array([v], np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, "value not exactly representable in bf16"
    return int(b >> 16)


# --------------------------------------------------------------------------- dequant
def test_dequant_golden_examples():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "dequant_examples.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for byte, elem, s, b, want in rows:
        q = np.zeros((1, 32), np.uint8)
        q[0, 0] = int(byte, 16)
        sc = np.full((1, 1), int(s, 16), np.uint16)
        bi = np.full((1, 1), int(b, 16), np.uint16)
        w = oracle.dequant(q, sc, bi, K=64)
        assert w[0, int(elem)] == float(want), (byte, elem, s, b)


def test_dequant_special_cases():
    rng = np.random.default_rng(0)
    rows, K = 8, 256
    s_vals = rng.uniform(0.005, 0.02, (rows, K // 64)).astype(np.float32)
    s_bits = (s_vals.view(np.uint32) >> 16).astype(np.uint16)          # truncation: still a bf16
    s = npr.bf16_to_f64(s_bits)
    # q = 0 -> bias exactly; q = 15 -> 15*s + b;  q = 8 with b = -8s -> 0 exactly
    b_bits = np.array([[_bf16_bits(-8.0 * float(v)) for v in row] for row in s], np.uint16)
    for qv, expect in ((0, lambda: npr.bf16_to_f64(b_bits)),
                       (15, lambda: 15 * s + npr.bf16_to_f64(b_bits)),
                       (8, lambda: np.zeros_like(s))):
        q = np.full((rows, K // 2), qv | (qv << 4), np.uint8)
        w = oracle.dequant(q, s_bits, b_bits, K=K)
        np.testing.assert_array_equal(w, np.repeat(expect(), 64, axis=1))


def test_dequant_pack_roundtrip_and_group_direction():
    rng = np.random.default_rng(1)
    rows, K = 5, 192
    vals = rng.integers(0, 16, (rows, K))
    packed = (vals[:, 0::2] | (vals[:, 1::2] << 4)).astype(np.uint8)
    one, zero = _bf16_bits(1.0), 0
    w = oracle.dequant(packed, np.full((rows, 3), one, np.uint16), np.full((rows, 3), zero, np.uint16), K=K)
    np.testing.assert_array_equal(w, vals.astype(np.float64))
    # distinct scale per group: group g of row n must use scale[n, g] (not [g, n], not k % 64)
    sc = np.array([[_bf16_bits(2.0 ** -(n + g)) for g in range(3)] for n in range(rows)], np.uint16)
    w = oracle.dequant(packed, sc, np.zeros((rows, 3), np.uint16), K=K)
    for n in range(rows):
        for g in range(3):
            np.testing.assert_array_equal(w[n, 64 * g:64 * (g + 1)], vals[n, 64 * g:64 * (g + 1)] * 2.0 ** -(n + g))


def test_dequant_matches_numpy_formulation():
    cfg = small_cfg()
    L, _ = small_layer(cfg)
    for n, K in (("gate", cfg.d), ("down", cfg.I)):
        np.testing.assert_array_equal(oracle.dequant(L[n + "_q"], L[n + "_s"], L[n + "_b"], K=K),
                                      npr.dequant(L[n + "_q"], L[n + "_s"], L[n + "_b"]))


# --------------------------------------------------------------------------- logits
def test_logits_match_library_matmul_and_bias():
    cfg = small_cfg(zipf_s=1.1)
    L, x = small_layer(cfg)
    lg = oracle.logits(x, L["router_w"], L["router_bias"])
    ref = npr.bf16_to_f64(x) @ npr.bf16_to_f64(L["router_w"]).T + L["router_bias"].astype(np.float64)
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-12)
    # one-hot activation picks one column of Wr (closed form, catches a transposed operand)
    d = cfg.d
    x1 = np.zeros((3, d), np.uint16)
    for t, c in enumerate((0, 5, d - 1)):
        x1[t, c] = _bf16_bits(1.0)
    lg1 = oracle.logits(x1, L["router_w"])
    for t, c in enumerate((0, 5, d - 1)):
        np.testing.assert_array_equal(lg1[t], npr.bf16_to_f64(L["router_w"][:, c]))


# --------------------------------------------------------------------------- selection
def test_select_worked_example_closed_form():
    # logits ln(1..8) on experts 0..7 and -10 elsewhere: the top 8 are 7,6,...,0
    # and the renormalised softmax weights are exactly n/36 (n = 8,...,1).
    E = 16
    lg = np.full((1, E), -10.0)
    lg[0, :8] = np.log(np.arange(1, 9))
    idx, w = oracle.select(lg, 8)
    assert idx[0].tolist() == [7, 6, 5, 4, 3, 2, 1, 0]
    np.testing.assert_allclose(w[0], np.arange(8, 0, -1) / 36.0, rtol=1e-14)


def test_select_ties_lower_index_first():
    E = 32
    lg = np.ones((2, E))
    lg[0, 7] = 2.0                      # one strict winner, then the seven lowest indices among ties
    lg[1, [30, 3, 17]] = 5.0            # a three-way tie at the top
    idx, w = oracle.select(lg, 8)
    assert idx[0].tolist() == [7, 0, 1, 2, 3, 4, 5, 6]
    e = math.e
    np.testing.assert_allclose(w[0], [e / (e + 7)] + [1 / (e + 7)] * 7, rtol=1e-14)
    assert idx[1].tolist() == [3, 17, 30, 0, 1, 2, 4, 5]


def test_select_zero_router_and_forced_bias():
    cfg = small_cfg(E=64, top_k=8)
    L, x = small_layer(cfg)
    zero = np.zeros_like(L["router_w"])
    idx, w = oracle.select(oracle.logits(x, zero), 8)
    assert (idx == np.arange(8)).all()
    assert (w == 0.125).all()
    forced = np.zeros(64, np.float32)
    chosen = [5, 9, 20, 33, 40, 41, 50, 63]
    forced[chosen] = 100.0
    idx, w = oracle.select(oracle.logits(x, L["router_w"], forced), 8)
    assert all(sorted(r) == chosen for r in idx.tolist())


def test_select_matches_full_softmax_renormalised():
    cfg = small_cfg(T=50, E=256, top_k=8)
    L, x = small_layer(cfg)
    lg = oracle.logits(x, L["router_w"])
    idx, w = oracle.select(lg, 8)
    ridx, rw = npr.select(lg, 8)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    assert all(len(set(r)) == 8 for r in idx.tolist())
    assert (np.diff(np.take_along_axis(lg, idx.astype(np.int64), 1), axis=1) <= 0).all()


# --------------------------------------------------------------------------- routing tables
def _check_tables(tab, idx, E, BM):
    T, k = idx.shape
    counts, offsets, perm, bm = tab["counts"], tab["offsets"], tab["perm"], tab["block_map"]
    # histogram: brute-force counting
    for e in range(E):
        assert counts[e] == int((idx == e).sum())
    assert counts.sum() == T * k
    # scan: monotone, 0 .. T*k
    assert offsets[0] == 0 and offsets[-1] == T * k and (np.diff(offsets) == counts).all()
    # scatter: a bijection on [0, T*k), each segment holds expert e in ascending token order
    assert sorted(perm.tolist()) == list(range(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (idx.reshape(-1)[seg] == e).all()
        assert (np.diff(seg // k) > 0).all()
    # block map: tiles every segment contiguously, no entry for empty experts
    assert tab["n_blocks"] == sum(-(-int(c) // BM) for c in counts)
    assert bm[:, 2].sum() == T * k and (bm[:, 2] >= 1).all() and (bm[:, 2] <= BM).all()
    cursor = {}
    for e, start, rows in bm.tolist():
        assert counts[e] > 0
        assert start == cursor.get(e, offsets[e])
        cursor[e] = start + rows
    assert all(cursor[e] == offsets[e + 1] for e in cursor)
    assert (np.diff(bm[:, 0]) >= 0).all()


@pytest.mark.parametrize("T,E,k,BM", [(1, 256, 8, 128), (37, 256, 8, 16), (300, 16, 4, 64), (0, 8, 2, 4)])
def test_route_tables_invariants_and_numpy(T, E, k, BM):
    rng = np.random.default_rng(T + E)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    tab = oracle.route_tables(idx, E, BM)
    _check_tables(tab, idx, E, BM)
    ref = npr.route_tables(idx, E, BM)
    for key in ("counts", "offsets", "perm", "block_map"):
        np.testing.assert_array_equal(tab[key], ref[key])


def test_route_tables_all_tokens_one_expert_set():
    T, E, k, BM = 260, 256, 8, 128
    idx = np.tile(np.arange(100, 108, dtype=np.int32), (T, 1))
    tab = oracle.route_tables(idx, E, BM)
    _check_tables(tab, idx, E, BM)
    assert tab["n_blocks"] == 8 * 3
    assert (tab["counts"][100:108] == T).all() and tab["counts"].sum() == T * k


# --------------------------------------------------------------------------- expert MLP + combine
def _moe(cfg, L, x, idx, w):
    return oracle.moe_tokens(L, x, idx, w, d=cfg.d, E=cfg.E, I=cfg.I, I_shared=cfg.I_shared)


def test_moe_matches_grouped_numpy_formulation():
    cfg = small_cfg()
    L, x = small_layer(cfg)
    idx, w = oracle.select(oracle.logits(x, L["router_w"]), cfg.top_k)
    out = _moe(cfg, L, x, idx, w)
    ref = npr.moe_layer(L, x, idx, w, E=cfg.E)
    assert rel_max_err(out, ref) < 1e-12
    # a token subset gives the same rows
    sub = oracle.moe_tokens(L, x, idx, w, [4, 1], d=cfg.d, E=cfg.E, I=cfg.I, I_shared=cfg.I_shared)
    np.testing.assert_array_equal(sub, out[[4, 1]])


def _const_q4(rows, K, qv, s, b):
    return (np.full((rows, K // 2), qv | (qv << 4), np.uint8),
            np.full((rows, K // 64), _bf16_bits(s), np.uint16), np.full((rows, K // 64), _bf16_bits(b), np.uint16))


def test_moe_constant_weights_closed_form():
    # All weights of one matrix equal one constant, so every expert is a scalar map:
    # g = cg*S, u = cu*S with S = sum(x); h = silu(g)*u; y = cd*I*h per output.
    cfg = small_cfg()
    d, I, E = cfg.d, cfg.I, cfg.E
    L, x = small_layer(cfg)
    consts = {"gate": (3, 2 ** -7, -2 ** -5), "up": (9, 2 ** -6, -2 ** -4), "down": (12, 2 ** -8, -2 ** -5)}
    for pre, scale_sh in (("", 1.0), ("sh_", 0.5)):
        for n, (qv, s, b) in consts.items():
            rows = (E if pre == "" else 1) * (I if n != "down" else d)
            K = d if n != "down" else I
            L[pre + n + "_q"], L[pre + n + "_s"], L[pre + n + "_b"] = _const_q4(rows, K, qv, s * scale_sh, b * scale_sh)
    idx, w = oracle.select(oracle.logits(x, L["router_w"]), cfg.top_k)
    out = _moe(cfg, L, x, idx, w)
    S = npr.bf16_to_f64(x).sum(1)

    def y(sc):
        cg = (3 * 2 ** -7 - 2 ** -5) * sc
        cu = (9 * 2 ** -6 - 2 ** -4) * sc
        cd = (12 * 2 ** -8 - 2 ** -5) * sc
        g, u = cg * S, cu * S
        return cd * I * (g / (1 + np.exp(-g))) * u

    expect = y(1.0) + y(0.5)                    # routed weights sum to 1; shared weight 1
    np.testing.assert_allclose(out, np.repeat(expect[:, None], d, 1), rtol=1e-12, atol=1e-12)


def test_moe_zero_weights_and_identical_experts():
    cfg = small_cfg()
    L, x = small_layer(cfg)
    d, I, E = cfg.d, cfg.I, cfg.E
    idx, w = oracle.select(oracle.logits(x, L["router_w"]), cfg.top_k)
    # identical routed experts: out = y_routed + y_shared for ANY routing, since sum(w) = 1
    L2 = dict(L)
    for n, R in (("gate", I), ("up", I), ("down", d)):
        for a in ("_q", "_s", "_b"):
            L2[n + a] = np.concatenate([L[n + a][:R]] * E)
    rng = np.random.default_rng(5)
    idx_rand = np.stack([rng.choice(E, cfg.top_k, replace=False) for _ in range(cfg.T)]).astype(np.int32)
    a = _moe(cfg, L2, x, idx, w)
    b = _moe(cfg, L2, x, idx_rand, w)
    assert rel_max_err(a, b) < 1e-12
    # all routed weights zero: only the shared expert remains
    L3 = dict(L)
    for n in ("gate", "up", "down"):
        L3[n + "_q"] = np.zeros_like(L[n + "_q"])
        L3[n + "_b"] = np.zeros_like(L[n + "_b"])
    shared_only = _moe(cfg, L3, x, idx, w)
    ref = npr.moe_layer(L3, x, idx, np.zeros_like(w), E=E)
    assert rel_max_err(shared_only, ref) < 1e-12
    # and with the shared expert zeroed too: exactly zero
    for n in ("sh_gate", "sh_up", "sh_down"):
        L3[n + "_q"] = np.zeros_like(L[n + "_q"])
        L3[n + "_b"] = np.zeros_like(L[n + "_b"])
    assert (_moe(cfg, L3, x, idx, w) == 0).all()


def test_silu_swiglu_orientation():
    # gate and up differ: silu must wrap the gate projection, not the up projection.
    cfg = small_cfg(T=2)
    d, I, E = cfg.d, cfg.I, cfg.E
    L, x = small_layer(cfg)
    for pre, rows_gu in (("", E * I), ("sh_", I)):
        L[pre + "gate_q"], L[pre + "gate_s"], L[pre + "gate_b"] = _const_q4(rows_gu, d, 0, 2 ** -7, -2 ** -3)
        L[pre + "up_q"], L[pre + "up_s"], L[pre + "up_b"] = _const_q4(rows_gu, d, 0, 2 ** -7, 2 ** -4)
        rows_d = E * d if pre == "" else d
        L[pre + "down_q"], L[pre + "down_s"], L[pre + "down_b"] = _const_q4(rows_d, I, 0, 2 ** -7, 2 ** -6)
    idx, w = oracle.select(oracle.logits(x, L["router_w"]), cfg.top_k)
    out = _moe(cfg, L, x, idx, w)
    S = npr.bf16_to_f64(x).sum(1)
    g, u = -S / 8, S / 16
    per_expert = 2 ** -6 * I * (g / (1 + np.exp(-g))) * u
    np.testing.assert_allclose(out[:, 0], 2 * per_expert, rtol=1e-12)


# --------------------------------------------------------------------------- decode chaining norm
def test_rms_norm_closed_form():
    out = np.array([[3.0, 4.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, 0.0]])
    xn = oracle.rms_norm(out, eps=0.0 + 1e-300)
    np.testing.assert_allclose(xn[0], np.array([3, 4, 0, 0]) / 2.5, rtol=1e-15)
    np.testing.assert_allclose(xn[1], 1.0, rtol=1e-15)
    assert (xn[2] == 0).all()
    xe = oracle.rms_norm(out[1:2], eps=3.0)
    np.testing.assert_allclose(xe, 0.5, rtol=1e-15)


# --------------------------------------------------------------------------- workload realism
@pytest.mark.slow
def test_zipf_workload_is_skewed():
    cfg = CONFIGS["prefill_t2048_zipf"]
    L = make_layer(cfg, "cpu")
    x = bits(make_x(cfg, "cpu"))
    lg = oracle.logits(x, bits(L["router_w"]), bits(L["router_bias"]))
    idx, _ = oracle.select(lg, cfg.top_k)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    assert (counts == 0).sum() >= 1
    assert (counts > 300).sum() >= 2
