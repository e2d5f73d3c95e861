"""Host-only checks of the C ABI: the library builds, loads and exports every
entry point declared in include/lily_moe.h, and argument validation returns the
documented codes before anything touches a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest
import torch

import bit_grouped_expert_top_gb300 as lm
from bit_grouped_expert_top_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lily_moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lily_moe_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = lm.load()
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value


def test_version_and_status_strings():
    assert lm.lily_moe_version() >= 10000
    for code in range(-9, 1):
        s = lm.lily_moe_status_string(code)
        assert s and s != "unknown status"
    assert lm.lily_moe_status_string(-99) == "unknown status"


def _shape(**kw):
    base = dict(T=512, d=2048)
    base.update(kw)
    return lm.make_shape(**base)


@pytest.mark.parametrize("kw,code", [
    ({}, 0), ({"T": 0}, 0), ({"T": 1}, 0), ({"d": 512, "I": 128}, 0), ({"block_rows": 16}, 0),
    ({"T": -1}, -1), ({"d": 0}, -1),
    ({"E": 128}, -2), ({"top_k": 4}, -2), ({"group": 32}, -2), ({"d": 2000}, -2), ({"I": 500}, -2),
    ({"I": 512, "I_shared": 1024}, -2), ({"block_rows": 256}, -2), ({"block_rows": 48}, -2),
])
def test_check_shape(kw, code):
    assert lm.lily_moe_check_shape(_shape(**kw)) == code


def test_block_capacity_and_workspace_sizes():
    s = _shape(T=512)
    assert lm.lily_moe_block_capacity(s) == min(512 * 8, 256 + 512 * 8 // 128)
    assert lm.lily_moe_block_capacity(_shape(T=1)) == 8
    assert lm.lily_moe_block_capacity(_shape(T=0)) == 1
    w512, w8192 = lm.lily_moe_workspace_bytes(s), lm.lily_moe_workspace_bytes(_shape(T=8192))
    assert 0 < w512 < w8192
    # h alone: (top_k + 1) * T * I bf16
    assert w8192 >= 9 * 8192 * 512 * 2
    assert lm.lily_moe_workspace_bytes(_shape(T=1), 40) >= lm.lily_moe_workspace_bytes(_shape(T=1))
    assert lm.lily_moe_workspace_bytes(_shape(T=9), 1) == 0          # decode needs T <= 8
    assert lm.lily_moe_workspace_bytes(_shape(E=64)) == 0


FAKE = 0x10000000  # an aligned address that is never dereferenced: validation fails first


def _fake_weights(misalign=None):
    w = _abi.lily_moe_weights()
    w.router_w = FAKE
    for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(w, n, _abi.lily_q4(FAKE, FAKE, FAKE))
    if misalign:
        setattr(w, misalign, _abi.lily_q4(FAKE + 2, FAKE, FAKE))
    return w


def _fake_routing(**kw):
    r = _abi.lily_moe_routing()
    for n, _ in r._fields_:
        setattr(r, n, FAKE)
    for k, v in kw.items():
        setattr(r, k, v)
    return r


def test_host_validation_codes_without_gpu():
    L = lm.load()
    s = _shape()
    need = lm.lily_moe_workspace_bytes(s)
    W, R = _fake_weights(), _fake_routing()
    by = ctypes.byref
    # null shape / weights / routing member
    assert L.lily_moe_route(None, by(W), FAKE, by(R), FAKE, need, None) == -1
    assert L.lily_moe_route(by(s), None, FAKE, by(R), FAKE, need, None) == -1
    assert L.lily_moe_route(by(s), by(W), FAKE, by(_fake_routing(perm=None)), FAKE, need, None) == -1
    # unsupported shape
    bad = _shape(E=64)
    assert L.lily_moe_forward(by(bad), by(W), FAKE, FAKE, None, FAKE, need, None) == -2
    # misaligned weight pointer, misaligned x, misaligned workspace (needs 256)
    assert L.lily_moe_forward(by(s), by(_fake_weights("down")), FAKE, FAKE, None, FAKE, need, None) == -3
    assert L.lily_moe_forward(by(s), by(W), FAKE + 8, FAKE, None, FAKE, need, None) == -3
    assert L.lily_moe_forward(by(s), by(W), FAKE, FAKE, None, FAKE + 16, need, None) == -3
    # workspace too small
    assert L.lily_moe_forward(by(s), by(W), FAKE, FAKE, None, FAKE, need - 1, None) == -4
    assert L.lily_moe_grouped_gemm(by(s), by(W), FAKE, by(R), FAKE, FAKE, 0, None) == -4
    # decode: T outside 1..8, zero layers, null layer array
    s9 = _shape(T=9)
    arr = (_abi.lily_moe_weights * 1)(W)
    assert L.lily_moe_decode(by(s9), 1, arr, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == -2
    s1 = _shape(T=1)
    assert L.lily_moe_decode(by(s1), 0, arr, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == -1
    assert L.lily_moe_decode(by(s1), 1, None, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == -1
    assert L.lily_moe_device_status(None, None) == -1


def test_zero_tokens_is_a_noop_without_gpu():
    L = lm.load()
    s = _shape(T=0)
    need = lm.lily_moe_workspace_bytes(s)
    W, R = _fake_weights(), _fake_routing()
    by = ctypes.byref
    assert L.lily_moe_route(by(s), by(W), None, by(R), FAKE, need, None) == 0
    assert L.lily_moe_grouped_gemm(by(s), by(W), None, by(R), None, FAKE, need, None) == 0
    assert L.lily_moe_forward(by(s), by(W), None, None, None, FAKE, need, None) == 0


def test_binding_rejects_host_tensors_before_calling_the_library():
    # a host tensor's address would reach the kernels as if it were device memory
    s = _shape(T=4)
    w = _fake_weights()
    r = _fake_routing()
    x_host = torch.zeros((4, 512), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.lily_moe_forward(s, w, x_host, FAKE, FAKE)
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.make_routing({"perm": torch.zeros(32, dtype=torch.int32)})
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.make_weights({k: torch.zeros(4) for k in ("router_w",)})
    with pytest.raises(ValueError, match="CUDA tensor"):
        lm.lily_moe_route(s, w, FAKE, r, torch.zeros(64, dtype=torch.uint8))


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_envelope_fits(T):
    # every decode shape of the documented envelope (T <= 8, d <= 4096, I <= 1024)
    # has a workspace size; larger d or I has none
    for d in (256, 512, 1024, 2048, 4096, 8192):
        for I in (128, 256, 512, 1024, 2048):
            s = _shape(T=T, d=d, I=I)
            want = d <= 4096 and I <= 1024
            assert (lm.lily_moe_workspace_bytes(s, 1) > 0) == want, (T, d, I)
