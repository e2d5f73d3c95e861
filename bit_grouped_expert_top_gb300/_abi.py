"""ctypes binding of liblily_moe.so (include/lily_moe.h), argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors are
passed as device pointers (``tensor.data_ptr()``), streams as the raw CUDA
stream handle of a ``torch.cuda.Stream`` (default: the current stream).  Every
step of the layer runs in the library's CUDA kernels; there is no Python or CPU
fallback: if the library cannot be loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Dict, Optional, Sequence

import torch

from . import build as _build

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

LILY_OK = 0
STATUS_NAMES = {0: "LILY_OK", -1: "LILY_ERR_INVALID", -2: "LILY_ERR_UNSUPPORTED", -3: "LILY_ERR_MISALIGNED",
                -4: "LILY_ERR_WORKSPACE", -5: "LILY_ERR_LAUNCH", -6: "LILY_ERR_DEVICE_TIMEOUT",
                -7: "LILY_ERR_DEVICE_INDEX", -8: "LILY_ERR_SCRATCH_LIMIT", -9: "LILY_ERR_DEVICE_RANGE"}


class LilyError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        detail = f"; {lily_moe_last_error_detail()}" if code == -5 else ""
        super().__init__(f"{fn} returned {code} ({STATUS_NAMES.get(code, '?')}: {lily_moe_status_string(code)}){detail}")


class lily_moe_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "d", "E", "top_k", "I", "I_shared", "group", "block_rows")]


class lily_q4(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class lily_moe_weights(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p)] + [
        (n, lily_q4) for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")]


class lily_moe_routing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "topk_idx", "topk_w", "counts", "offsets", "perm", "block_map", "n_blocks")]


class lily_attn_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "H_q", "H_kv", "D", "block_size", "max_blocks")]


class lily_gdn_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H_k", "H_v", "d_k", "d_v")]


class lily_moe_decode_trace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("logits", "topk_idx", "topk_w")]


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declares the argument and return types of every entry point."""
    P, S, I32, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64
    PS, PW, PR = ctypes.POINTER(lily_moe_shape), ctypes.POINTER(lily_moe_weights), ctypes.POINTER(lily_moe_routing)
    L.lily_moe_version.restype = I32
    L.lily_moe_status_string.restype = ctypes.c_char_p
    L.lily_moe_status_string.argtypes = [I32]
    L.lily_moe_last_error_detail.restype = ctypes.c_char_p
    L.lily_moe_last_error_detail.argtypes = []
    L.lily_moe_check_shape.argtypes = [PS]
    L.lily_moe_block_capacity.restype = I64
    L.lily_moe_block_capacity.argtypes = [PS]
    L.lily_moe_workspace_bytes.restype = S
    L.lily_moe_workspace_bytes.argtypes = [PS, ctypes.c_int32]
    L.lily_moe_route.argtypes = [PS, PW, P, PR, P, S, P]
    L.lily_moe_grouped_gemm.argtypes = [PS, PW, P, PR, P, P, S, P]
    L.lily_moe_forward.argtypes = [PS, PW, P, P, PR, P, S, P]
    L.lily_moe_forward_timed.argtypes = [PS, PW, P, P, PR, P, S, P, ctypes.POINTER(ctypes.c_void_p)]
    L.lily_moe_decode.argtypes = [PS, ctypes.c_int32, PW, P, P, P, ctypes.POINTER(lily_moe_decode_trace), P, S, P]
    L.lily_moe_route_noalloc.argtypes = [PS, PW, P, PR, P, P]
    PA = ctypes.POINTER(lily_attn_shape)
    L.lily_attn_workspace_bytes.restype = S
    L.lily_attn_workspace_bytes.argtypes = [PA]
    L.lily_attn_decode.argtypes = [PA, P, P, P, I64, P, P, ctypes.c_float, P, P, S, P]
    L.lily_attn_decode.restype = I32
    L.lily_gdn_scan.argtypes = [ctypes.POINTER(lily_gdn_shape), P, P, P, P, P, P, ctypes.c_float, P, P, P]
    L.lily_gdn_scan.restype = I32
    L.lily_moe_device_status.argtypes = [P, P]
    L.lily_moe_clear_status.argtypes = [P, P]
    for n in ("lily_moe_check_shape", "lily_moe_route", "lily_moe_grouped_gemm", "lily_moe_forward",
              "lily_moe_forward_timed", "lily_moe_decode", "lily_moe_device_status", "lily_moe_route_noalloc",
              "lily_moe_clear_status"):
        getattr(L, n).restype = I32
    return L


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads the in-tree library (building it first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.build()
            if not os.path.exists(p):
                raise OSError(f"liblily_moe.so not found at {p}")
            _lib = _configure(ctypes.CDLL(p))
    return _lib


_variants: Dict[str, ctypes.CDLL] = {}


def load_variant(variant: str) -> ctypes.CDLL:
    """Loads a test-only build variant of the library (see build.VARIANTS) as a
    separate library with its own kernels and static device data."""
    with _lock:
        if variant not in _variants:
            _variants[variant] = _configure(ctypes.CDLL(_build.build(variants=(variant,))))
    return _variants[variant]


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t) -> Optional[int]:
    """Device address of a tensor argument (None stays NULL; an int is taken as a
    raw device pointer).  Tensors must be dense CUDA tensors: the library reads
    them as row-major device arrays and cannot tell a host address from a device one."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device} (shape {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {t.stride()} (shape {tuple(t.shape)})")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc != LILY_OK:
        raise LilyError(fn, rc)
    return rc


def make_shape(T: int, d: int, E: int = 256, top_k: int = 8, I: int = 512, I_shared: Optional[int] = None,
               group: int = 64, block_rows: int = 128) -> lily_moe_shape:
    return lily_moe_shape(T, d, E, top_k, I, I if I_shared is None else I_shared, group, block_rows)


def make_weights(layer: Dict[str, torch.Tensor]) -> lily_moe_weights:
    """Weight struct of one layer from a dict of device tensors (names as in
    bit_grouped_expert_top_gb300.inputs.make_layer).  The caller keeps the
    tensors alive."""
    w = lily_moe_weights()
    w.router_w = _ptr(layer["router_w"])
    w.router_bias = _ptr(layer.get("router_bias"))
    for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(w, n, lily_q4(_ptr(layer[n + "_q"]), _ptr(layer[n + "_s"]), _ptr(layer[n + "_b"])))
    return w


def make_routing(tensors: Dict[str, torch.Tensor]) -> lily_moe_routing:
    r = lily_moe_routing()
    for n, _ in lily_moe_routing._fields_:
        setattr(r, n, _ptr(tensors.get(n)))
    return r


def alloc_routing(shape: lily_moe_shape, device="cuda", with_logits: bool = True) -> Dict[str, torch.Tensor]:
    """Caller-owned routing tables for `shape` (torch allocates them)."""
    T, E, k = shape.T, shape.E, shape.top_k
    cap = lily_moe_block_capacity(shape)
    out = {
        "topk_idx": torch.empty((T, k), dtype=torch.int32, device=device),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device=device),
        "counts": torch.empty((E,), dtype=torch.int32, device=device),
        "offsets": torch.empty((E + 1,), dtype=torch.int32, device=device),
        "perm": torch.empty((T * k,), dtype=torch.int32, device=device),
        "block_map": torch.empty((max(cap, 1), 3), dtype=torch.int32, device=device),
        "n_blocks": torch.empty((1,), dtype=torch.int32, device=device),
    }
    if with_logits:
        out["logits"] = torch.empty((T, E), dtype=torch.float32, device=device)
    return out


def alloc_workspace(shape: lily_moe_shape, n_layers_decode: int = 0, device="cuda") -> torch.Tensor:
    n = lily_moe_workspace_bytes(shape, n_layers_decode)
    if n == 0:
        raise LilyError("lily_moe_workspace_bytes", -2)
    ws = torch.zeros((n,), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


# ------------------------------------------------------------------ entry points (same names as the C ABI)
def lily_moe_version() -> int:
    return load().lily_moe_version()


def lily_moe_status_string(code: int) -> str:
    return load().lily_moe_status_string(int(code)).decode()


def lily_moe_last_error_detail() -> str:
    return load().lily_moe_last_error_detail().decode()


def lily_moe_check_shape(shape: lily_moe_shape) -> int:
    return load().lily_moe_check_shape(ctypes.byref(shape))


def lily_moe_block_capacity(shape: lily_moe_shape) -> int:
    return load().lily_moe_block_capacity(ctypes.byref(shape))


def lily_moe_workspace_bytes(shape: lily_moe_shape, n_layers_decode: int = 0) -> int:
    return load().lily_moe_workspace_bytes(ctypes.byref(shape), int(n_layers_decode))


def lily_moe_route(shape, weights, x, routing, ws, stream=None, *, check: bool = True) -> int:
    rc = load().lily_moe_route(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), ctypes.byref(routing),
                               _ptr(ws), ws.numel() if isinstance(ws, torch.Tensor) else 0, _stream(stream))
    return _check("lily_moe_route", rc) if check else rc


def lily_moe_grouped_gemm(shape, weights, x, routing, out, ws, stream=None, *, check: bool = True) -> int:
    rc = load().lily_moe_grouped_gemm(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), ctypes.byref(routing),
                                      _ptr(out), _ptr(ws), ws.numel() if isinstance(ws, torch.Tensor) else 0,
                                      _stream(stream))
    return _check("lily_moe_grouped_gemm", rc) if check else rc


def lily_moe_forward(shape, weights, x, out, ws, routing=None, stream=None, *, check: bool = True) -> int:
    rc = load().lily_moe_forward(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(out),
                                 None if routing is None else ctypes.byref(routing), _ptr(ws),
                                 ws.numel() if isinstance(ws, torch.Tensor) else 0, _stream(stream))
    return _check("lily_moe_forward", rc) if check else rc


def lily_moe_forward_timed(shape, weights, x, out, ws, events: Sequence[torch.cuda.Event], routing=None,
                           stream=None, *, check: bool = True) -> int:
    """As lily_moe_forward, recording 6 events (start, after router GEMM, after
    routing tables, after the routing-order copy of x, after gate/up, after down)."""
    assert len(events) == 6
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on first record
            e.record(torch.cuda.current_stream() if stream is None else stream)
    arr = (ctypes.c_void_p * 6)(*[e.cuda_event for e in events])
    rc = load().lily_moe_forward_timed(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), _ptr(out),
                                       None if routing is None else ctypes.byref(routing), _ptr(ws),
                                       ws.numel() if isinstance(ws, torch.Tensor) else 0, _stream(stream), arr)
    return _check("lily_moe_forward_timed", rc) if check else rc


def lily_moe_decode(shape, layers: Sequence[lily_moe_weights], x, out, ws, x_next=None,
                    trace: Optional[Dict[str, torch.Tensor]] = None, stream=None, *, check: bool = True) -> int:
    arr = (lily_moe_weights * len(layers))(*layers)
    tr = None
    if trace is not None:
        tr = lily_moe_decode_trace(_ptr(trace.get("logits")), _ptr(trace.get("topk_idx")), _ptr(trace.get("topk_w")))
    rc = load().lily_moe_decode(ctypes.byref(shape), len(layers), arr, _ptr(x), _ptr(out), _ptr(x_next),
                                None if tr is None else ctypes.byref(tr), _ptr(ws),
                                ws.numel() if isinstance(ws, torch.Tensor) else 0, _stream(stream))
    return _check("lily_moe_decode", rc) if check else rc


def lily_moe_device_status(ws, stream=None) -> int:
    return load().lily_moe_device_status(_ptr(ws), _stream(stream))


def lily_moe_clear_status(ws, stream=None) -> int:
    return _check("lily_moe_clear_status", load().lily_moe_clear_status(_ptr(ws), _stream(stream)))


def lily_moe_route_noalloc(shape, weights, x, routing, device_status=None, stream=None, *, check: bool = True) -> int:
    """Routing without a caller workspace: for callers that may not allocate
    device memory when they run the layer (e.g. inside another engine's fixed
    memory budget).  Scratch lives in a fixed device array owned by the
    library (T <= 8192); calls that may overlap on the GPU race.  `routing`
    must include logits; `device_status` (device int32 tensor) receives the
    call's device status."""
    rc = load().lily_moe_route_noalloc(ctypes.byref(shape), ctypes.byref(weights), _ptr(x), ctypes.byref(routing),
                                       _ptr(device_status), _stream(stream))
    return _check("lily_moe_route_noalloc", rc) if check else rc


# ------------------------------------------------------------------ decode attention
def make_attn_shape(B: int, H_q: int, H_kv: int, D: int, block_size: int, max_blocks: int) -> lily_attn_shape:
    return lily_attn_shape(B, H_q, H_kv, D, block_size, max_blocks)


def lily_attn_workspace_bytes(shape: lily_attn_shape) -> int:
    return load().lily_attn_workspace_bytes(ctypes.byref(shape))


def alloc_attn_workspace(shape: lily_attn_shape, device="cuda") -> torch.Tensor:
    n = lily_attn_workspace_bytes(shape)
    if n == 0:
        raise ValueError("unsupported attention shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def lily_attn_decode(shape: lily_attn_shape, q, k_cache, v_cache, block_table, seq_lens, out, ws,
                     scale: Optional[float] = None, stream=None, *, check: bool = True) -> int:
    """Grouped-query decode attention over a fixed-block KV cache (see
    include/lily_moe.h).  scale defaults to 1/sqrt(D)."""
    if scale is None:
        scale = 1.0 / math.sqrt(shape.D)
    n_blocks = k_cache.shape[0] if isinstance(k_cache, torch.Tensor) else 0
    rc = load().lily_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), n_blocks,
                                 _ptr(block_table), _ptr(seq_lens), float(scale), _ptr(out), _ptr(ws),
                                 ws.numel() if isinstance(ws, torch.Tensor) else 0, _stream(stream))
    return _check("lily_attn_decode", rc) if check else rc


# ------------------------------------------------------------------ Gated DeltaNet scan
def lily_gdn_scan(q, k, v, alpha, beta, out, state_out, state_in=None, scale: Optional[float] = None,
                  stream=None, *, check: bool = True) -> int:
    """Gated DeltaNet scan over the T tokens of q/k [T][H_k][d_k], v [T][H_v][d_v]
    (see include/lily_moe.h).  scale defaults to 1/sqrt(d_k)."""
    T, H_k, d_k = q.shape
    _, H_v, d_v = v.shape
    shape = lily_gdn_shape(T, H_k, H_v, d_k, d_v)
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    rc = load().lily_gdn_scan(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(state_in),
                              float(scale), _ptr(out), _ptr(state_out), _stream(stream))
    return _check("lily_gdn_scan", rc) if check else rc
