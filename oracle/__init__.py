"""fp64 CPU oracle of the mixture-of-experts layer, of grouped-query decode
attention over a fixed-block KV cache and of the Gated DeltaNet scan: ctypes
wrappers around oracle.c.

TEST INFRASTRUCTURE ONLY.  Only tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never calls it and
it never calls the CUDA library; the two share no code.

All array arguments are numpy arrays.  bf16 tensors are passed as their uint16
bit patterns; packed 4-bit weights as uint8 [rows, K/2] (low nibble = even k).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, fp64, OpenMP).  Returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("d", "E", "I", "I_shared", "G")] + [
        (n, ctypes.c_void_p) for n in (
            "gate_q", "up_q", "down_q",
            "gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b",
            "sh_gate_q", "sh_up_q", "sh_down_q",
            "sh_gate_s", "sh_gate_b", "sh_up_s", "sh_up_b", "sh_down_s", "sh_down_b")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.oracle_num_threads.restype = I32
            L.oracle_set_threads.argtypes = [I32]
            L.oracle_dequant.argtypes = [P, P, P, I64, I64, I64, P]
            L.oracle_logits.argtypes = [P, P, P, I64, I64, I64, P]
            L.oracle_select.argtypes = [P, I64, I64, I64, P, P]
            L.oracle_route_tables.argtypes = [P, I64, I64, I64, I64, P, P, P, P, P]
            L.oracle_moe_tokens.argtypes = [ctypes.POINTER(OracleLayer), P, I64, P, P, P, I64, P]
            L.oracle_rms_norm.argtypes = [P, I64, I64, ctypes.c_double, P]
            L.oracle_attn_decode.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I64, ctypes.c_double, P]
            L.oracle_gdn_scan.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, ctypes.c_double, P, P]
            _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def dequant(q: np.ndarray, scale: np.ndarray, bias: np.ndarray, K: int, group: int = 64) -> np.ndarray:
    """w[n, k] = q[n, k] * scale[n, k // group] + bias[n, k // group]  (fp64)."""
    q, scale, bias = _c(q, np.uint8), _c(scale, np.uint16), _c(bias, np.uint16)
    rows = q.shape[0]
    assert q.shape == (rows, K // 2) and scale.shape == (rows, K // group) == bias.shape
    w = np.empty((rows, K), np.float64)
    lib().oracle_dequant(_p(q), _p(scale), _p(bias), rows, K, group, _p(w))
    return w


def logits(x: np.ndarray, wr: np.ndarray, bias_r: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t, e] = sum_k x[t, k] * Wr[e, k] + bias_r[e]  (fp64, from bf16 bits)."""
    x, wr = _c(x, np.uint16), _c(wr, np.uint16)
    T, d = x.shape
    E = wr.shape[0]
    b = None if bias_r is None else _c(bias_r, np.float32)
    out = np.empty((T, E), np.float64)
    lib().oracle_logits(_p(x), _p(wr), _p(b), T, d, E, _p(out))
    return out


def select(lg: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k experts per token (descending logit, lower index first on ties) and
    their renormalised softmax weights.  Float32 logits are widened exactly."""
    lg = _c(lg, np.float64)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().oracle_select(_p(lg), T, E, k, _p(idx), _p(w))
    return idx, w


def route_tables(idx: np.ndarray, E: int, block_rows: int):
    """Histogram, exclusive scan, stable scatter and block map of a selection."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    nmax = max(1, min(T * k, E + -(-T * k // block_rows)))
    bm = np.zeros((nmax, 3), np.int32)
    nb = np.zeros(1, np.int32)
    lib().oracle_route_tables(_p(idx), T, E, k, block_rows, _p(counts), _p(offsets),
                              _p(perm), _p(bm), _p(nb))
    return {"counts": counts, "offsets": offsets, "perm": perm,
            "block_map": bm[: int(nb[0])].copy(), "n_blocks": int(nb[0])}


_WEIGHT_NAMES = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")


def _layer_struct(layer: Dict[str, np.ndarray], d: int, E: int, I: int, I_shared: int, group: int):
    keep = {}
    st = OracleLayer(d=d, E=E, I=I, I_shared=I_shared, G=group)
    for n in _WEIGHT_NAMES:
        q = keep[n + "_q"] = _c(layer[n + "_q"], np.uint8)
        s = keep[n + "_s"] = _c(layer[n + "_s"], np.uint16)
        b = keep[n + "_b"] = _c(layer[n + "_b"], np.uint16)
        setattr(st, n + "_q", q.ctypes.data)
        setattr(st, n + "_s", s.ctypes.data)
        setattr(st, n + "_b", b.ctypes.data)
    return st, keep


def moe_tokens(layer: Dict[str, np.ndarray], x: np.ndarray, idx: np.ndarray, w: np.ndarray,
               tokens: Optional[Sequence[int]] = None, *, d: int, E: int, I: int,
               I_shared: int, group: int = 64) -> np.ndarray:
    """out[t] = sum_j w[t, j] * SwiGLU_{idx[t, j]}(x_t) + SwiGLU_shared(x_t), fp64,
    for the listed tokens (all tokens if None).  Returns [len(tokens), d]."""
    x = _c(x, np.uint16)
    idx = _c(idx, np.int32)
    w = _c(w, np.float64)
    T, k = idx.shape
    toks = np.arange(T, dtype=np.int64) if tokens is None else _c(np.asarray(tokens), np.int64)
    st, keep = _layer_struct(layer, d, E, I, I_shared, group)
    out = np.empty((len(toks), d), np.float64)
    lib().oracle_moe_tokens(ctypes.byref(st), _p(x), k, _p(idx), _p(w), _p(toks), len(toks), _p(out))
    del keep
    return out


def rms_norm(out: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """xn[t] = out[t] / sqrt(mean(out[t]^2) + eps)."""
    out = _c(out, np.float64)
    T, d = out.shape
    xn = np.empty_like(out)
    lib().oracle_rms_norm(_p(out), T, d, eps, _p(xn))
    return xn


def attn_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_table: np.ndarray,
                seq_lens: np.ndarray, scale: Optional[float] = None) -> np.ndarray:
    """Grouped-query decode attention over a fixed-block KV cache, fp64.

    q: bf16 bits [B][H_q][D]; k_cache, v_cache: bf16 bits [n_blocks][H_kv][bs][D];
    block_table: int32 [B][max_blocks]; seq_lens: int32 [B].  Returns [B][H_q][D]
    doubles: o_h = sum_t softmax_t(scale q_h . k_{g,t}) v_{g,t}, g = h / (H_q / H_kv).
    """
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, H_q, D = q.shape
    n_blocks, H_kv, bs, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and H_q % H_kv == 0
    assert block_table.shape[0] == B and seq_lens.shape == (B,)
    assert int(seq_lens.max(initial=0)) <= block_table.shape[1] * bs
    used = np.concatenate([block_table[b, :(int(seq_lens[b]) + bs - 1) // bs] for b in range(B)])
    assert used.size == 0 or (used.min() >= 0 and used.max() < n_blocks)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((B, H_q, D), np.float64)
    lib().oracle_attn_decode(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(seq_lens), B, H_q, H_kv, D, bs,
                             block_table.shape[1], float(scale), _p(out))
    return out


def gdn_scan(q: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray,
             S0: Optional[np.ndarray] = None, scale: float = 1.0) -> Tuple[np.ndarray, np.ndarray]:
    """Gated DeltaNet scan over T tokens, fp64.

    q, k: bf16 bits [T][H_k][d_k]; v: bf16 bits [T][H_v][d_v]; alpha, beta: f32
    [T][H_v]; S0: [H_v][d_v][d_k] or None (zeros).  Returns (o [T][H_v][d_v],
    S_T [H_v][d_v][d_k]) with S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t
    S_{t-1} k_t) k_t^T and o_t = scale S_t q_t.
    """
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    alpha, beta = _c(alpha, np.float32), _c(beta, np.float32)
    T, H_k, dk = q.shape
    T2, H_v, dv = v.shape
    assert k.shape == q.shape and T2 == T and H_v % H_k == 0
    assert alpha.shape == (T, H_v) and beta.shape == (T, H_v)
    if S0 is not None:
        S0 = _c(S0, np.float64)
        assert S0.shape == (H_v, dv, dk)
    o = np.empty((T, H_v, dv), np.float64)
    S = np.empty((H_v, dv, dk), np.float64)
    lib().oracle_gdn_scan(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(S0), T, H_k, H_v, dk, dv, float(scale),
                          _p(o), _p(S))
    return o, S
