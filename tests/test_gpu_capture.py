"""The entry points enqueue only stream work, so a caller may record them into
its own CUDA graph: each call is captured on a side stream, the outputs are
poisoned, and one replay must write what a direct call wrote (bit for bit, or,
for the prefill layer, whose combine adds in arrival order, to fp32 rounding)."""
import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
from bit_grouped_expert_top_gb300.attn_inputs import ATTN_CONFIGS, make_attn
from bit_grouped_expert_top_gb300.gdn_inputs import GDN_CONFIGS, make_gdn
from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x
from gpu_util import Layer, shape_of, x_for

pytestmark = pytest.mark.gpu


def _replay_matches(fn, outs, exact=True):
    fn(torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    for o in outs:
        o.fill_(float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn(side)
    torch.cuda.synchronize()
    assert all(bool(torch.isnan(o).all()) for o in outs), "capture must not run the work"
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        if exact:
            assert torch.equal(a, b)
        else:
            scale = float(a.abs().max())
            assert float((a - b).abs().max()) <= 1e-6 * max(scale, 1.0)


def test_attention_capture():
    cfg = ATTN_CONFIGS["attn_tiny"]
    a = {k: v.cuda() for k, v in make_attn(cfg, "cpu", 0).items()}
    s = lm.make_attn_shape(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.block_size, cfg.max_blocks)
    ws = lm.alloc_attn_workspace(s)
    out = torch.empty((cfg.B, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
    _replay_matches(lambda st: lm.lily_attn_decode(s, a["q"], a["k_cache"], a["v_cache"], a["block_table"],
                                                   a["seq_lens"], out, ws, stream=st), [out])
    assert lm.lily_moe_device_status(ws) == 0


def test_gdn_capture():
    g = {k: v.cuda() for k, v in make_gdn(GDN_CONFIGS["gdn_tiny"]).items()}
    out = torch.empty(g["v"].shape, dtype=torch.float32, device="cuda")
    st = torch.empty_like(g["state"])
    _replay_matches(lambda s: lm.lily_gdn_scan(g["q"], g["k"], g["v"], g["alpha"], g["beta"], out, st,
                                               state_in=g["state"], stream=s), [out, st])


def test_forward_capture():
    cfg = CONFIGS["tiny"]
    w = lm.make_weights(layer := make_layer(cfg, "cuda"))
    x = make_x(cfg, "cuda")
    s = lm.make_shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I, I_shared=cfg.I_shared,
                      group=cfg.group, block_rows=cfg.block_rows)
    ws = lm.alloc_workspace(s)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    _replay_matches(lambda st: lm.lily_moe_forward(s, w, x, out, ws, stream=st), [out], exact=False)
    assert lm.lily_moe_device_status(ws) == 0
    del layer


def test_decode_capture():
    # a capturing stream gets the launches directly instead of the cached graph
    cfg = CONFIGS["tiny"]
    layers = [Layer(cfg, layer_index=l) for l in range(2)]
    s = shape_of(cfg, 2)
    ws = lm.alloc_workspace(s, n_layers_decode=2)
    x = x_for(cfg, T=2, seed_offset=102)
    out = torch.empty((2, 2, cfg.d), dtype=torch.float32, device="cuda")
    x_next = torch.empty((2, 2, cfg.d), dtype=torch.bfloat16, device="cuda")
    _replay_matches(lambda st: lm.lily_moe_decode(s, [L.w for L in layers], x, out, ws, x_next=x_next, stream=st),
                    [out])
    assert lm.lily_moe_device_status(ws) == 0
