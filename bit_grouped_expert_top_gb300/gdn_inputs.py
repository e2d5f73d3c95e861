"""Seeded synthetic inputs for the Gated DeltaNet scan.

Like `inputs.py`, this module only draws random numbers; the recurrence itself
lives in the CUDA kernel and in the fp64 oracle, which share nothing else.

Workload recipe (the linear-attention layers of a Qwen3.6-35B-A3B-style model:
the page "Perplexity libera o Lily" on noticiai.com.br, section "O modelo em
tres formatos de carga", gives 30 Gated DeltaNet layers with a fixed-size
state; head counts and sizes are not on the page; the reading here is the
hybrid Qwen models' 16 query/key heads and 32 value heads of size 128):

* q, k: bf16 random unit vectors per head (the layer normalises them before
  the scan); v: bf16 N(0, 1)
* decay alpha: f32 U[0.9, 1.0]; write strength beta: f32 U[0, 1]
* initial state: f32 N(0, 0.05^2) (a prefill chunk continuing a sequence), or
  zeros
* scale: 1 / sqrt(d_k)
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict

import torch


@dataclass(frozen=True)
class GDNConfig:
    name: str
    T: int
    H_k: int = 16
    H_v: int = 32
    d_k: int = 128
    d_v: int = 128
    seed: int = 0
    with_state: bool = True

    def with_(self, **kw) -> "GDNConfig":
        return replace(self, **kw)


GDN_CONFIGS: Dict[str, GDNConfig] = {
    "gdn_tiny": GDNConfig("gdn_tiny", T=37, H_k=2, H_v=4, d_k=64, d_v=64, seed=21),
    "gdn_t512": GDNConfig("gdn_t512", T=512, seed=22),
    "gdn_t8192": GDNConfig("gdn_t8192", T=8192, seed=23),
}


def _unit(shape, g, device) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device)
    return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)


def make_gdn(cfg: GDNConfig, device="cpu") -> Dict[str, torch.Tensor]:
    g = torch.Generator(device=device)
    g.manual_seed(7727 * (cfg.seed + 1))
    out = {
        "q": _unit((cfg.T, cfg.H_k, cfg.d_k), g, device),
        "k": _unit((cfg.T, cfg.H_k, cfg.d_k), g, device),
        "v": torch.randn((cfg.T, cfg.H_v, cfg.d_v), generator=g, device=device).to(torch.bfloat16),
        "alpha": torch.rand((cfg.T, cfg.H_v), generator=g, device=device) * 0.1 + 0.9,
        "beta": torch.rand((cfg.T, cfg.H_v), generator=g, device=device),
    }
    if cfg.with_state:
        out["state"] = torch.randn((cfg.H_v, cfg.d_v, cfg.d_k), generator=g, device=device) * 0.05
    return out


def gdn_bytes(cfg: GDNConfig) -> int:
    """Bytes a scan reads and writes once: q, k, v, alpha, beta, the state in and
    out, and the f32 output."""
    T = cfg.T
    return (2 * T * cfg.H_k * cfg.d_k * 2 + T * cfg.H_v * cfg.d_v * 2 + 2 * T * cfg.H_v * 4
            + 2 * cfg.H_v * cfg.d_v * cfg.d_k * 4 + T * cfg.H_v * cfg.d_v * 4)


def gdn_flops(cfg: GDNConfig) -> int:
    """Per token and value head: S k (2 d_v d_k), the update (2 d_v d_k) and S q
    (2 d_v d_k)."""
    return 6 * cfg.T * cfg.H_v * cfg.d_v * cfg.d_k
