"""Seeded synthetic inputs for grouped-query decode attention over a fixed-block
KV cache.

Like `inputs.py`, this module only draws random numbers and lays them out; it
holds none of the attention arithmetic, so the CUDA path and the fp64 oracle
can both be fed from it.

Workload recipe (the full-attention layers of a Qwen3.6-35B-A3B-style model:
the page "Perplexity libera o Lily" on noticiai.com.br, section "O modelo em
tres formatos de carga", gives 16 query heads and two KV heads over a growing
KV cache; section "Prefill e decode" measures decode at 32K, 64K and 128K
tokens of context and names a fixed-block cache layout):

* q, K, V: bf16, N(0, 1)
* head dimension D (256 for the measured workloads: the page gives no size;
  256 is the head size of the hybrid-attention Qwen models with 16 query and
  2 KV heads)
* cache blocks of `block_size` tokens, layout [block][kv head][row][D]; each
  sequence's logical blocks map to physical blocks through a seeded random
  permutation (so a sequence's blocks are not contiguous in the cache)
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Tuple

import torch


@dataclass(frozen=True)
class AttnConfig:
    """Shape and seed of one synthetic decode-attention workload."""

    name: str
    seq_lens: Tuple[int, ...]  # tokens in the cache of each sequence (B = len)
    H_q: int = 16
    H_kv: int = 2
    D: int = 256
    block_size: int = 64
    seed: int = 0
    n_sets: int = 1            # distinct caches cycled by the benchmark

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def max_blocks(self) -> int:
        return max((L + self.block_size - 1) // self.block_size for L in self.seq_lens)

    def with_(self, **kw) -> "AttnConfig":
        return replace(self, **kw)


ATTN_CONFIGS: Dict[str, AttnConfig] = {
    # three sequences (one token, a ragged block, several blocks): the oracle is instant
    "attn_tiny": AttnConfig("attn_tiny", seq_lens=(1, 100, 777), D=128, seed=11),
    # batch-1 decode at the page's three context lengths
    "attn_32k": AttnConfig("attn_32k", seq_lens=(32768,), seed=12, n_sets=4),
    "attn_64k": AttnConfig("attn_64k", seq_lens=(65536,), seed=13, n_sets=2),
    "attn_128k": AttnConfig("attn_128k", seq_lens=(131072,), seed=14),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_attn(cfg: AttnConfig, device="cpu", set_index: int = 0, extra_blocks: int = 3) -> Dict[str, torch.Tensor]:
    """q [B][H_q][D], k_cache / v_cache [n_blocks][H_kv][block_size][D] (bf16),
    block_table [B][max_blocks] and seq_lens [B] (int32).  Unused table entries
    are -1; the cache holds `extra_blocks` blocks no sequence uses."""
    g = _gen(device, 9973 * (cfg.seed + 1) + 613 * set_index)
    nb = [(L + cfg.block_size - 1) // cfg.block_size for L in cfg.seq_lens]
    n_blocks = sum(nb) + extra_blocks
    q = torch.randn((cfg.B, cfg.H_q, cfg.D), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((n_blocks, cfg.H_kv, cfg.block_size, cfg.D), generator=g, device=device).to(torch.bfloat16)
    v = torch.randn((n_blocks, cfg.H_kv, cfg.block_size, cfg.D), generator=g, device=device).to(torch.bfloat16)
    phys = torch.randperm(n_blocks, generator=g, device=device).to(torch.int32)
    table = torch.full((cfg.B, cfg.max_blocks), -1, dtype=torch.int32, device=device)
    at = 0
    for b, n in enumerate(nb):
        table[b, :n] = phys[at:at + n]
        at += n
    lens = torch.tensor(cfg.seq_lens, dtype=torch.int32, device=device)
    return {"q": q, "k_cache": k, "v_cache": v, "block_table": table, "seq_lens": lens}


def kv_bytes(cfg: AttnConfig) -> int:
    """Bytes of K and V one decode step reads: every cached token of every KV head."""
    return 2 * cfg.H_kv * sum(cfg.seq_lens) * cfg.D * 2
