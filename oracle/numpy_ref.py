"""A second, vectorised fp64 formulation of the MoE layer in numpy.

TEST INFRASTRUCTURE ONLY.  It exists to pin the C oracle: where the C oracle
walks token by token and element by element, this module uses library
primitives (matmul, stable argsort, bincount, cumsum) and computes the experts
grouped in expert-sorted order.  The two agree only if both follow the same
definition (the page "Perplexity libera o Lily", sections "O modelo em tres
formatos de carga" and "Prefill e decode").
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def unpack_nibbles(q: np.ndarray) -> np.ndarray:
    """uint8 [rows, K/2] -> int [rows, K]; low nibble is the even element."""
    q = np.asarray(q, np.uint8)
    lo = q & 0x0F
    hi = q >> 4
    return np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1).astype(np.int64)


def dequant(q, scale, bias, group: int = 64) -> np.ndarray:
    qv = unpack_nibbles(q).astype(np.float64)
    s = np.repeat(bf16_to_f64(scale), group, axis=1)
    b = np.repeat(bf16_to_f64(bias), group, axis=1)
    return qv * s + b


def logits(x_bits, wr_bits, bias_r: Optional[np.ndarray] = None) -> np.ndarray:
    lg = bf16_to_f64(x_bits) @ bf16_to_f64(wr_bits).T
    if bias_r is not None:
        lg = lg + np.asarray(bias_r, np.float32).astype(np.float64)[None, :]
    return lg


def select(lg: np.ndarray, k: int):
    """Softmax over all E, keep the k largest (stable sort: lower index first on
    equal logits), renormalise over the k kept."""
    lg = np.asarray(lg, np.float64)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    pk = np.take_along_axis(p, order, axis=1)
    return order.astype(np.int32), pk / pk.sum(axis=1, keepdims=True)


def route_tables(idx: np.ndarray, E: int, block_rows: int):
    idx = np.asarray(idx, np.int64)
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    perm = np.argsort(flat, kind="stable")
    bm = []
    for e in range(E):
        for start in range(0, int(counts[e]), block_rows):
            bm.append((e, int(offsets[e]) + start, min(block_rows, int(counts[e]) - start)))
    bm = np.array(bm, np.int64).reshape(-1, 3)
    return {"counts": counts, "offsets": offsets, "perm": perm, "block_map": bm,
            "n_blocks": len(bm)}


def silu(z):
    return z / (1.0 + np.exp(-z))


def moe_layer(layer: Dict[str, np.ndarray], x_bits, idx, w, *, E: int, group: int = 64) -> np.ndarray:
    """Grouped formulation: sort assignments by expert, run each expert once on
    its gathered rows, scale by the routing weight and add back in token order;
    then add the shared expert with weight 1."""
    x = bf16_to_f64(x_bits)
    T, d = x.shape
    idx = np.asarray(idx, np.int64)
    w = np.asarray(w, np.float64)
    k = idx.shape[1]
    I = layer["gate_q"].shape[0] // E
    out = np.zeros((T, d))

    def mlp(xs, gq, gs, gb, uq, us, ub, dq, ds, db):
        Wg, Wu, Wd = dequant(gq, gs, gb, group), dequant(uq, us, ub, group), dequant(dq, ds, db, group)
        return (silu(xs @ Wg.T) * (xs @ Wu.T)) @ Wd.T

    tabs = route_tables(idx, E, block_rows=1 << 30)
    for e in range(E):
        lo, hi = tabs["offsets"][e], tabs["offsets"][e + 1]
        if hi == lo:
            continue
        a = tabs["perm"][lo:hi]
        toks, slots = a // k, a % k
        r, rd = slice(e * I, (e + 1) * I), slice(e * d, (e + 1) * d)
        y = mlp(x[toks], layer["gate_q"][r], layer["gate_s"][r], layer["gate_b"][r],
                layer["up_q"][r], layer["up_s"][r], layer["up_b"][r],
                layer["down_q"][rd], layer["down_s"][rd], layer["down_b"][rd])
        np.add.at(out, toks, w[toks, slots][:, None] * y)
    out += mlp(x, layer["sh_gate_q"], layer["sh_gate_s"], layer["sh_gate_b"],
               layer["sh_up_q"], layer["sh_up_s"], layer["sh_up_b"],
               layer["sh_down_q"], layer["sh_down_s"], layer["sh_down_b"])
    return out
