"""Shared test plumbing: torch <-> numpy conversion and small synthetic layers."""
from __future__ import annotations

from typing import Dict

import numpy as np
import torch

from bit_grouped_expert_top_gb300.inputs import LayerConfig, make_layer, make_x


def bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's uint16 bit patterns (any other dtype: plain numpy)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def layer_np(layer: Dict[str, torch.Tensor]) -> Dict[str, np.ndarray]:
    return {k: bits(v) for k, v in layer.items()}


def small_cfg(**kw) -> LayerConfig:
    """A layer small enough for pure-numpy cross-checks on CPU."""
    base = dict(name="small", T=6, d=128, E=16, top_k=4, I=64, I_shared=64, seed=11)
    base.update(kw)
    return LayerConfig(**base)


def small_layer(cfg: LayerConfig):
    return layer_np(make_layer(cfg, "cpu")), bits(make_x(cfg, "cpu"))


def rel_max_err(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.square(ref))))
    return float(np.max(np.abs(a - ref))) / max(rms, 1e-300)
