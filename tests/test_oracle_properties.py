"""Property pins of the fp64 oracle's routing on random inputs (hypothesis).

Selection (page "Perplexity libera o Lily", noticiai.com.br, section "O modelo
em tres formatos de carga": a router scores the experts and keeps eight): the
oracle's top-k must equal a brute-force full sort of (-logit, expert) pairs,
even on rows full of equal logits, and its weights must be the softmax over the
kept logits.  Routing tables (section "Prefill e decode": histogram, prefix
scan, scatter, block map): on random shapes, skews and tile heights the tables
must satisfy every invariant and match the vectorised numpy formulation.
"""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import numpy_ref as npr  # noqa: E402
from test_oracle import _check_tables  # noqa: E402


@st.composite
def logit_rows(draw):
    E = draw(st.sampled_from([8, 16, 64, 256]))
    k = draw(st.integers(1, min(8, E)))
    T = draw(st.integers(1, 12))
    tie_heavy = draw(st.booleans())
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    if tie_heavy:  # a handful of distinct values: many equal logits per row
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float64)
    else:
        lg = rng.standard_normal((T, E)) * draw(st.sampled_from([1e-3, 1.0, 30.0]))
    return lg, k


@settings(max_examples=150, deadline=None)
@given(logit_rows())
def test_select_equals_brute_force_sort_and_softmax(case):
    lg, k = case
    idx, w = oracle.select(lg, k)
    T, E = lg.shape
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))[:k]
        assert idx[t].tolist() == order
        kept = [lg[t, e] for e in order]
        m = max(kept)
        den = sum(math.exp(v - m) for v in kept)
        np.testing.assert_allclose(w[t], [math.exp(v - m) / den for v in kept], rtol=1e-13, atol=0)
        assert abs(float(np.sum(w[t])) - 1.0) < 1e-12


@st.composite
def routings(draw):
    E = draw(st.sampled_from([4, 8, 16, 64, 256]))
    k = draw(st.integers(1, min(8, E)))
    T = draw(st.integers(0, 300))
    BM = draw(st.sampled_from([1, 4, 16, 64, 128]))
    skew = draw(st.sampled_from([0.0, 1.0, 3.0]))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    # k distinct experts per token, drawn with Zipf-like preferences when skewed
    pref = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
    keys = rng.random((T, E)) ** (1.0 / pref)  # larger preference -> keys nearer 1
    idx = np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    return idx.reshape(T, k), E, BM


@settings(max_examples=150, deadline=None)
@given(routings())
def test_route_tables_invariants_on_random_routings(case):
    idx, E, BM = case
    tab = oracle.route_tables(idx, E, BM)
    _check_tables(tab, idx, E, BM)
    ref = npr.route_tables(idx, E, BM)
    for key in ("counts", "offsets", "perm", "block_map"):
        np.testing.assert_array_equal(tab[key], ref[key])
