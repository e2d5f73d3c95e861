"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and the
fp64 oracle on the same seeded inputs."""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np
import torch

import bit_grouped_expert_top_gb300 as lm
import oracle
from oracle import numpy_ref as npr
from bit_grouped_expert_top_gb300.inputs import LayerConfig, make_layer, make_x
from helpers import bits, layer_np

# Output bound of the layer: max|gpu - oracle| <= 1e-2 * rms(oracle)
# (the rebuilt weights, x and h rounded to fp16 inside the GPU path, fp32
# accumulation).
OUT_TOL = 1e-2
# Router logits: bf16 x bf16 products are exact in fp32; the fp32 sums are not.
# A sum of K products, added in at most D rounded steps along any path, is off
# from the exact value by at most D * 2^-24 * sum_k |x_k w_k| (first order).
# D = K/8 + 64 covers the tensor core's K/16 chained MMAs (plus its adds inside
# one MMA) and the CUDA-core GEMVs (at most 64 sequential adds per lane, then
# the warp and block reductions); the bias add is one more rounding.
LOGIT_TOL = 1e-5  # identical computations (two entry points over the same kernels)


def logit_error_bound(x_bits: np.ndarray, wr_bits: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Per-logit bound [T, E] of the fp32 accumulation error (see above)."""
    xa = np.abs(npr.bf16_to_f64(np.asarray(x_bits)))
    wa = np.abs(npr.bf16_to_f64(np.asarray(wr_bits)))
    K = xa.shape[1]
    u = 2.0 ** -24
    b = (K // 8 + 64) * u * (xa @ wa.T)
    if bias is not None:
        b = b + 2 * u * np.abs(np.asarray(bias, np.float64))[None, :]
    return b + 1e-30


def shape_of(cfg: LayerConfig, T: Optional[int] = None):
    return lm.make_shape(T=cfg.T if T is None else T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I,
                         I_shared=cfg.I_shared, group=cfg.group, block_rows=cfg.block_rows)


class Layer:
    """One layer's weights on the GPU (+ their numpy copy on demand)."""

    def __init__(self, cfg: LayerConfig, layer_index: int = 0, overrides: Optional[Dict[str, torch.Tensor]] = None):
        self.cfg = cfg
        self.t = make_layer(cfg, "cuda", layer_index)
        if overrides:
            self.t.update({k: v.cuda() for k, v in overrides.items()})
        self.w = lm.make_weights(self.t)
        self._np = None

    @property
    def np(self):
        if self._np is None:
            self._np = layer_np(self.t)
        return self._np


GUARD_BYTES = 4096
GUARD_BYTE = 0xA5


class Guarded:
    """Device tensors allocated with a GUARD_BYTES tail of GUARD_BYTE after
    them; check() asserts that no kernel wrote past the end of any of them."""

    def __init__(self):
        self.bufs = {}

    def empty(self, name: str, shape, dtype) -> torch.Tensor:
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((n + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
        self.bufs[name] = (raw, n)
        return raw[:n].view(dtype).view(shape)

    def check(self):
        for name, (raw, n) in self.bufs.items():
            tail = raw[n:].cpu().numpy()
            assert np.all(tail == GUARD_BYTE), f"{name}: {int(np.sum(tail != GUARD_BYTE))} guard bytes overwritten"


def run_forward(cfg: LayerConfig, layer: Layer, x: torch.Tensor, block_rows: Optional[int] = None,
                poison_workspace: bool = False):
    """lily_moe_forward through the C ABI with caller-owned routing tables.
    Every output buffer carries a guard tail that is checked afterwards; with
    poison_workspace the workspace starts as all-ones bytes (NaN as floats,
    -1 as integers) apart from the cleared status word."""
    T = x.shape[0]
    s = shape_of(cfg, T)
    if block_rows is not None:
        s.block_rows = block_rows
    ws = lm.alloc_workspace(s)
    if poison_workspace:
        ws.fill_(0xFF)
        lm.lily_moe_clear_status(ws)
    g = Guarded()
    cap = max(lm.lily_moe_block_capacity(s), 1)
    E, k = cfg.E, cfg.top_k
    rt = {"logits": g.empty("logits", (T, E), torch.float32),
          "topk_idx": g.empty("topk_idx", (T, k), torch.int32),
          "topk_w": g.empty("topk_w", (T, k), torch.float32),
          "counts": g.empty("counts", (E,), torch.int32),
          "offsets": g.empty("offsets", (E + 1,), torch.int32),
          "perm": g.empty("perm", (T * k,), torch.int32),
          "block_map": g.empty("block_map", (cap, 3), torch.int32),
          "n_blocks": g.empty("n_blocks", (1,), torch.int32)}
    r = lm.make_routing(rt)
    out = g.empty("out", (T, cfg.d), torch.float32)
    lm.lily_moe_forward(s, layer.w, x, out, ws, routing=r)
    status = lm.lily_moe_device_status(ws)
    assert status == 0, lm.lily_moe_status_string(status)
    torch.cuda.synchronize()
    g.check()
    res = {k: v.cpu().numpy() for k, v in rt.items()}
    res["out"] = out.cpu().numpy()
    res["n_blocks"] = int(res["n_blocks"][0])
    res["block_map"] = res["block_map"][: res["n_blocks"]]
    return res


def oracle_layer_out(cfg: LayerConfig, layer: Layer, x_bits: np.ndarray, gpu_logits: np.ndarray,
                     tokens: Optional[Sequence[int]] = None) -> np.ndarray:
    """Oracle output given the GPU's fp32 logits (same routing decisions)."""
    idx, w = oracle.select(gpu_logits.astype(np.float64), cfg.top_k)
    return oracle.moe_tokens(layer.np, x_bits, idx, w, tokens, d=cfg.d, E=cfg.E, I=cfg.I, I_shared=cfg.I_shared,
                             group=cfg.group)


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, tol: float = OUT_TOL):
    rms = float(np.sqrt(np.mean(np.square(ref))))
    err = float(np.max(np.abs(gpu.astype(np.float64) - ref)))
    assert np.isfinite(gpu).all()
    assert err <= tol * rms, f"max|gpu-oracle| = {err:.3e} > {tol} * rms {rms:.3e} (ratio {err / rms:.3e})"
    return err / rms


def assert_routing_exact(cfg: LayerConfig, res: Dict[str, np.ndarray], block_rows: Optional[int] = None):
    """Selection, histogram, scan, scatter and block map equal the oracle's
    run on the GPU's own fp32 logits, bit for bit; weights to fp32 rounding."""
    lg = res["logits"].astype(np.float64)
    idx, w = oracle.select(lg, cfg.top_k)
    np.testing.assert_array_equal(res["topk_idx"], idx)
    np.testing.assert_allclose(res["topk_w"], w, rtol=0, atol=2e-6)
    tab = oracle.route_tables(idx, cfg.E, block_rows or cfg.block_rows)
    for key in ("counts", "offsets", "perm", "block_map"):
        np.testing.assert_array_equal(res[key], tab[key], err_msg=key)
    assert res["n_blocks"] == tab["n_blocks"]


def assert_logits_close(cfg: LayerConfig, layer: Layer, x_bits: np.ndarray, gpu_logits: np.ndarray,
                        tokens: Optional[Sequence[int]] = None):
    xs = x_bits if tokens is None else x_bits[np.asarray(tokens)]
    gl = gpu_logits if tokens is None else gpu_logits[np.asarray(tokens)]
    ref = oracle.logits(xs, layer.np["router_w"], layer.np.get("router_bias"))
    bound = logit_error_bound(xs, layer.np["router_w"], layer.np.get("router_bias"))
    ratio = np.abs(gl.astype(np.float64) - ref) / bound
    assert float(ratio.max()) <= 1.0, f"logits error {float(ratio.max()):.2f} x the fp32 accumulation bound"


def sample_tokens(T: int, n: int, seed: int = 0):
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, T - 1), size=min(n, T - 2), replace=False) if T > 2 else np.array([], int)
    return np.unique(np.concatenate([[0, T - 1], mid])).astype(np.int64)


def x_for(cfg: LayerConfig, T: Optional[int] = None, seed_offset: int = 0) -> torch.Tensor:
    return make_x(cfg, "cuda", seed_offset=seed_offset, T=T)
