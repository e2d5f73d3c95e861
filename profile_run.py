"""Runs a few whole-layer forward passes of one seeded workload, for profilers
(a fixed, short launch sequence to put under ncu).

  python profile_run.py --config prefill_t8192 --reps 2
  python profile_run.py --config decode_t1_l40 --layers 4 --T 1 --reps 3
  python profile_run.py --config attn_32k --reps 4
  python profile_run.py --config gdn_t512 --reps 3

Each pass launches, in order: router GEMM, top-8 + per-chunk counts, per-expert
scan + block map, scatter, prep (fp16 x in routing order), gate/up GEMM +
SwiGLU (which also zeroes out), down GEMM + weighted combine.  An attention
config (attn_*) runs lily_attn_decode: split kernel, then combine kernel; a
gdn_* config runs lily_gdn_scan (one kernel).
Exits non-zero if the device status word reports an error.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import torch  # noqa: E402

import bit_grouped_expert_top_gb300 as lm  # noqa: E402
from bit_grouped_expert_top_gb300.attn_inputs import ATTN_CONFIGS, make_attn  # noqa: E402
from bit_grouped_expert_top_gb300.gdn_inputs import GDN_CONFIGS, make_gdn  # noqa: E402
from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x  # noqa: E402


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="prefill_t2048_zipf", choices=sorted(CONFIGS) + sorted(ATTN_CONFIGS) + sorted(GDN_CONFIGS))
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--layers", type=int, default=4, help="decode: distinct layers per call")
    ap.add_argument("--T", type=int, default=1, help="decode: tokens")
    a = ap.parse_args(argv)
    if a.config in ATTN_CONFIGS:
        return run_attention(ATTN_CONFIGS[a.config], a)
    if a.config in GDN_CONFIGS:
        return run_gdn(GDN_CONFIGS[a.config], a)
    cfg = CONFIGS[a.config]
    if a.config.startswith("decode"):
        return run_decode(cfg, a)
    layer = make_layer(cfg, "cuda")
    w = lm.make_weights(layer)
    x = make_x(cfg, "cuda")
    s = lm.make_shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I, I_shared=cfg.I_shared,
                      group=cfg.group, block_rows=cfg.block_rows)
    ws = lm.alloc_workspace(s)
    out = torch.empty((cfg.T, cfg.d), device="cuda")
    for _ in range(a.reps):
        lm.lily_moe_forward(s, w, x, out, ws)
    torch.cuda.synchronize()
    st = lm.lily_moe_device_status(ws)
    print(f"{a.config}: {a.reps} forward passes, device status {st}")
    return 0 if st == 0 else 1


def run_decode(cfg, a) -> int:
    layers = [make_layer(cfg, "cuda", i) for i in range(a.layers)]
    wl = [lm.make_weights(x) for x in layers]
    s = lm.make_shape(T=a.T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I, I_shared=cfg.I_shared,
                      group=cfg.group, block_rows=cfg.block_rows)
    ws = lm.alloc_workspace(s, n_layers_decode=a.layers)
    x = make_x(cfg, "cuda", T=a.T)
    out = torch.empty((a.layers, a.T, cfg.d), device="cuda")
    for _ in range(a.reps):
        lm.lily_moe_decode(s, wl, x, out, ws)
    torch.cuda.synchronize()
    st = lm.lily_moe_device_status(ws)
    print(f"{cfg.name}: {a.reps} decode calls of {a.layers} layers at T={a.T}, device status {st}")
    return 0 if st == 0 else 1


def run_attention(cfg, a) -> int:
    t = {k: v.cuda() for k, v in make_attn(cfg, "cpu").items()}
    s = lm.make_attn_shape(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.block_size, cfg.max_blocks)
    ws = lm.alloc_attn_workspace(s)
    out = torch.empty((cfg.B, cfg.H_q, cfg.D), device="cuda")
    for _ in range(a.reps):
        lm.lily_attn_decode(s, t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_lens"], out, ws)
    torch.cuda.synchronize()
    st = lm.lily_moe_device_status(ws)
    print(f"{cfg.name}: {a.reps} decode-attention calls, device status {st}")
    return 0 if st == 0 else 1


def run_gdn(cfg, a) -> int:
    g = {k: v.cuda() for k, v in make_gdn(cfg, "cpu").items()}
    out = torch.empty((cfg.T, cfg.H_v, cfg.d_v), device="cuda")
    st = torch.empty((cfg.H_v, cfg.d_v, cfg.d_k), device="cuda")
    for _ in range(a.reps):
        lm.lily_gdn_scan(g["q"], g["k"], g["v"], g["alpha"], g["beta"], out, st, state_in=g.get("state"))
    torch.cuda.synchronize()
    ok = bool(torch.isfinite(out).all())
    print(f"{cfg.name}: {a.reps} scans of {cfg.T} tokens, finite output {ok}")
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())
