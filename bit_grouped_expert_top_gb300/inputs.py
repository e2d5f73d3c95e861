"""Seeded synthetic inputs for the mixture-of-experts layer.

This module only draws random numbers.  It holds none of the layer's arithmetic
(no dequantisation, no routing, no GEMM), so the CUDA path and the fp64 oracle
can both be fed from it without sharing any of the method.

Workload recipe (one Qwen3.6-35B-A3B-style MoE layer; the page "Perplexity
libera o Lily" on noticiai.com.br, section "O modelo em tres formatos de carga",
gives 256 routed experts, top-8 and one shared expert; section "Prefill e
decode" gives the 4-bit group-64 affine weight format with bf16 scale and bias):

* activations x: bf16, N(0, 1)
* router weight Wr [E, d]: bf16, N(0, 1/d)   (variance 1/d)
* packed weights q: uniform random bytes, so every nibble is uniform on 0..15
* scale: bf16, U[0.005, 0.02]
* bias:  bf16(-8 * scale + N(0, 1e-3))       (std 1e-3)
* skewed routing: an additive router bias  bias_r[e] = -s * ln(rank_e)  with
  rank a seeded permutation of 1..E, which makes expert loads roughly Zipf(s).

Layouts (row-major, little-endian):
* q    : uint8 [rows, K/2], element k of a row in byte k/2, LOW nibble = even k
* scale, bias : bf16 [rows, K/64]
* routed experts are stacked by expert: gate/up rows = E*I (K = d),
  down rows = E*d (K = I); the shared expert has its own arrays.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Dict, Optional

import torch


@dataclass(frozen=True)
class LayerConfig:
    """Shape and seed of one synthetic MoE-layer workload."""

    name: str
    T: int                 # tokens
    d: int                 # hidden size
    E: int = 256           # routed experts
    top_k: int = 8
    I: int = 512           # routed-expert intermediate size
    I_shared: int = 512    # shared-expert intermediate size
    group: int = 64        # quantisation group along the reduction dim
    block_rows: int = 128  # rows per block-map entry
    seed: int = 0
    zipf_s: Optional[float] = None  # additive router bias for skewed loads
    n_weight_sets: int = 1          # distinct layer weight sets cycled
    n_layers: int = 1               # decode: layers run back to back

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# The five workloads the layer is measured and checked on.
CONFIGS: Dict[str, LayerConfig] = {
    # T=32, d=512, I=128: small enough for the oracle to finish in seconds.
    "tiny": LayerConfig("tiny", T=32, d=512, I=128, I_shared=128, seed=0),
    # The 512-token prefill point.
    "prefill_t512": LayerConfig("prefill_t512", T=512, d=2048, seed=1),
    # Skewed expert loads at T=2048 (Zipf s=1.1 router bias).
    "prefill_t2048_zipf": LayerConfig("prefill_t2048_zipf", T=2048, d=2048, seed=2, zipf_s=1.1),
    # Large prefill; 4 weight sets cycled so weights stream from HBM.
    "prefill_t8192": LayerConfig("prefill_t8192", T=8192, d=2048, seed=3, n_weight_sets=4),
    # Batch-1 decode over 40 distinct layers (also swept at T=2, 4, 8).
    "decode_t1_l40": LayerConfig("decode_t1_l40", T=1, d=2048, seed=4, n_layers=40),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _bf16_normal(shape, std: float, g, device) -> torch.Tensor:
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def _q4(rows: int, K: int, g, device) -> torch.Tensor:
    return torch.randint(0, 256, (rows, K // 2), generator=g, device=device, dtype=torch.uint8)


def _scale_bias(rows: int, K: int, group: int, g, device):
    ng = K // group
    scale = (torch.rand((rows, ng), generator=g, device=device) * 0.015 + 0.005).to(torch.bfloat16)
    noise = torch.randn((rows, ng), generator=g, device=device) * 1e-3
    bias = (-8.0 * scale.float() + noise).to(torch.bfloat16)
    return scale, bias


def make_x(cfg: LayerConfig, device="cpu", seed_offset: int = 0, T: Optional[int] = None) -> torch.Tensor:
    """Activations x [T, d] bf16 ~ N(0, 1)."""
    g = _gen(device, 1000003 * (cfg.seed + 1) + 17 + seed_offset)
    return _bf16_normal((cfg.T if T is None else T, cfg.d), 1.0, g, device)


def make_layer(cfg: LayerConfig, device="cpu", layer_index: int = 0) -> Dict[str, torch.Tensor]:
    """One layer's weights as a dict of tensors (names follow the C-ABI fields)."""
    g = _gen(device, 7919 * (cfg.seed + 1) + 104729 * layer_index)
    E, d, I, Is, G = cfg.E, cfg.d, cfg.I, cfg.I_shared, cfg.group
    w: Dict[str, torch.Tensor] = {}
    w["router_w"] = _bf16_normal((E, d), 1.0 / math.sqrt(d), g, device)
    if cfg.zipf_s is not None:
        rank = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        w["router_bias"] = (-cfg.zipf_s * torch.log(rank)).to(torch.float32)
    for name, rows, K in (("gate", E * I, d), ("up", E * I, d), ("down", E * d, I),
                          ("sh_gate", Is, d), ("sh_up", Is, d), ("sh_down", d, Is)):
        w[name + "_q"] = _q4(rows, K, g, device)
        w[name + "_s"], w[name + "_b"] = _scale_bias(rows, K, G, g, device)
    return w


def weight_bytes(cfg: LayerConfig) -> Dict[str, int]:
    """Bytes of each weight kind of one layer (int4 payload plus bf16 scale and bias)."""
    d, I, G = cfg.d, cfg.I, cfg.group
    per_matrix = d * I // 2 + 2 * 2 * (d * I // G)
    return {"expert": 3 * per_matrix, "router": cfg.E * d * 2,
            "layer": (cfg.E + 1) * 3 * per_matrix + cfg.E * d * 2}
