"""Pins of the fp64 Gated DeltaNet scan oracle (page "Perplexity libera o Lily",
sections "O modelo em tres formatos de carga" and "Prefill e decode": a
fixed-size recurrence scanned with its state in registers; the reading is the
gated delta rule S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,
o_t = scale S_t q_t) against closed forms of special cases, the delta rule's
retrieval property, linearity, and the product form of the recurrence."""
import numpy as np
import torch

import oracle
from bit_grouped_expert_top_gb300.gdn_inputs import GDN_CONFIGS, make_gdn


def bits(a) -> np.ndarray:
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def val(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand(rng, T=6, H_k=2, H_v=4, dk=8, dv=5):
    q = bits(rng.standard_normal((T, H_k, dk)))
    k = bits(rng.standard_normal((T, H_k, dk)) / np.sqrt(dk))
    v = bits(rng.standard_normal((T, H_v, dv)))
    a = rng.uniform(0.5, 1.0, (T, H_v)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, (T, H_v)).astype(np.float32)
    S0 = rng.standard_normal((H_v, dv, dk)) * 0.3
    return q, k, v, a, b, S0


def test_no_write_no_decay_keeps_the_state():
    # alpha = 1, beta = 0: S_t = S0 and o_t = scale S0 q_t
    rng = np.random.default_rng(1)
    q, k, v, a, b, S0 = _rand(rng)
    a[:] = 1.0
    b[:] = 0.0
    o, S = oracle.gdn_scan(q, k, v, a, b, S0, scale=0.5)
    np.testing.assert_array_equal(S, S0)
    for t in range(q.shape[0]):
        for h in range(4):
            np.testing.assert_allclose(o[t, h], 0.5 * S0[h] @ val(q[t, h // 2]), rtol=1e-14, atol=1e-14)


def test_full_decay_keeps_only_the_last_write():
    # alpha = 0: S_t = beta_t v_t k_t^T, o_t = scale beta_t v_t (k_t . q_t)
    rng = np.random.default_rng(2)
    q, k, v, a, b, S0 = _rand(rng)
    a[:] = 0.0
    o, S = oracle.gdn_scan(q, k, v, a, b, S0)
    for t in range(q.shape[0]):
        for h in range(4):
            kk, qq = val(k[t, h // 2]), val(q[t, h // 2])
            np.testing.assert_allclose(o[t, h], float(b[t, h]) * val(v[t, h]) * (kk @ qq), rtol=1e-13, atol=1e-14)
    T = q.shape[0]
    for h in range(4):
        np.testing.assert_allclose(S[h], float(b[T - 1, h]) * np.outer(val(v[T - 1, h]), val(k[T - 1, h // 2])),
                                   rtol=1e-13, atol=1e-14)


def test_orthonormal_keys_write_one_column_each():
    # alpha = beta = 1, S0 = 0, k_t = e_t: the delta rule stores v_t in column t,
    # so o_t = scale sum_{i <= t} v_i q_t[i]
    rng = np.random.default_rng(3)
    T, dk, dv = 6, 8, 5
    q, k, v, a, b, _ = _rand(rng, T=T, H_k=1, H_v=1, dk=dk, dv=dv)
    k[:] = 0
    for t in range(T):
        k[t, 0] = bits(np.eye(dk)[t])
    a[:] = 1.0
    b[:] = 1.0
    o, S = oracle.gdn_scan(q, k, v, a, b, None, scale=2.0)
    for t in range(T):
        ref = 2.0 * sum(val(v[i, 0]) * val(q[t, 0])[i] for i in range(t + 1))
        np.testing.assert_allclose(o[t, 0], ref, rtol=1e-14, atol=1e-14)


def test_delta_rule_retrieves_the_last_value():
    # beta = 1 and a unit key (0.5, 0.5, 0.5, 0.5): after the write S_T k_T = v_T,
    # whatever the state before it and the decay
    rng = np.random.default_rng(4)
    q, k, v, a, b, S0 = _rand(rng, H_k=1, H_v=1, dk=4, dv=3)
    T = q.shape[0]
    k[T - 1, 0] = bits([0.5, 0.5, 0.5, 0.5])
    b[T - 1, 0] = 1.0
    _, S = oracle.gdn_scan(q, k, v, a, b, S0)
    np.testing.assert_allclose(S[0] @ val(k[T - 1, 0]), val(v[T - 1, 0]), rtol=1e-13, atol=1e-13)


def test_linear_in_values_and_initial_state():
    # for fixed q, k, alpha, beta the scan is linear in (v, S0); small integer values
    # keep v1 + v2 exact in bf16
    rng = np.random.default_rng(5)
    q, k, _, a, b, S1 = _rand(rng)
    v1 = bits(rng.integers(-8, 9, (6, 4, 5)))
    v2 = bits(rng.integers(-8, 9, (6, 4, 5)))
    vs = bits(val(v1) + val(v2))
    assert np.array_equal(val(vs), val(v1) + val(v2))
    S2 = rng.standard_normal(S1.shape) * 0.3
    o1, T1 = oracle.gdn_scan(q, k, v1, a, b, S1)
    o2, T2 = oracle.gdn_scan(q, k, v2, a, b, S2)
    o3, T3 = oracle.gdn_scan(q, k, vs, a, b, S1 + S2)
    np.testing.assert_allclose(o3, o1 + o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(T3, T1 + T2, rtol=1e-12, atol=1e-12)


def test_matches_the_product_form():
    # S_T = S0 A_1 ... A_T + sum_t beta_t v_t k_t^T A_{t+1} ... A_T with
    # A_t = alpha_t (I - beta_t k_t k_t^T), and o_t = scale S_t q_t (numpy matrices)
    rng = np.random.default_rng(6)
    q, k, v, a, b, S0 = _rand(rng, T=7, H_k=1, H_v=2, dk=6, dv=4)
    o, S = oracle.gdn_scan(q, k, v, a, b, S0, scale=0.7)
    T, dk = 7, 6
    for h in range(2):
        A = [float(a[t, h]) * (np.eye(dk) - float(b[t, h]) * np.outer(val(k[t, 0]), val(k[t, 0]))) for t in range(T)]
        for t in range(T):
            St = S0[h].copy()
            for s in range(t + 1):
                St = St @ A[s]
            for s in range(t + 1):
                W = float(b[s, h]) * np.outer(val(v[s, h]), val(k[s, 0]))
                for r in range(s + 1, t + 1):
                    W = W @ A[r]
                St = St + W
            np.testing.assert_allclose(o[t, h], 0.7 * St @ val(q[t, 0]), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(S[h], St, rtol=1e-11, atol=1e-12)


def test_value_heads_share_their_key_head():
    # value heads 2h and 2h + 1 read key head h: with equal inputs they agree
    rng = np.random.default_rng(7)
    q, k, v, a, b, S0 = _rand(rng)
    v[:, 1] = v[:, 0]
    a[:, 1] = a[:, 0]
    b[:, 1] = b[:, 0]
    S0[1] = S0[0]
    o, S = oracle.gdn_scan(q, k, v, a, b, S0)
    np.testing.assert_array_equal(o[:, 1], o[:, 0])
    assert np.abs(o[:, 2] - o[:, 0]).max() > 0


def test_generated_workload_shapes():
    c = GDN_CONFIGS["gdn_tiny"]
    g = make_gdn(c)
    assert g["q"].shape == (c.T, c.H_k, c.d_k) and g["v"].shape == (c.T, c.H_v, c.d_v)
    n = g["k"].float().norm(dim=-1)
    assert float((n - 1).abs().max()) < 1e-2
