"""The C-ABI library builds, loads and exports every function the header declares;
host-side argument checks answer without touching a GPU."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "sparse_expert_swiglu.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def so():
    from sparse_expert_swiglu_gb300 import build
    path = build.build()
    return path


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["moe_route_topk", "expert_pack_int2_up", "moe_expert_sparse_swiglu",
                     "moe_layer_decode", "moe_layer_workspace_bytes", "moe_get_status",
                     "moe_status_string", "expert_unpack_int2_up"]:
        assert required in names


def test_library_exports_every_declared_symbol(so):
    handle = ctypes.CDLL(so)
    for name in _declared_functions():
        assert hasattr(handle, name), name


def test_binding_covers_the_header(so):
    from sparse_expert_swiglu_gb300 import _lib
    assert set(_lib.EXPORTED) == set(_declared_functions())


def test_library_has_no_torch_dependency(so):
    with open(so, "rb") as fh:
        data = fh.read()
    assert b"libtorch" not in data and b"c10::" not in data


def test_status_strings(so):
    from sparse_expert_swiglu_gb300 import _lib
    lib = _lib.lib()
    assert lib.moe_status_string(0) == b"ok"
    assert lib.moe_status_string(-2) == b"unsupported shape"
    assert lib.moe_status_string(-6) == b"device-side wait timed out"


def test_packed_size(so):
    from sparse_expert_swiglu_gb300 import _lib
    lib = _lib.lib()
    assert lib.expert_int2_up_packed_bytes(4096, 14336) == (14336 // 16) * 8 * 2560
    # 0.3125 bytes per weight when d is a multiple of 512
    assert lib.expert_int2_up_packed_bytes(4096, 14336) == 4096 * 14336 * 5 // 16
    assert lib.expert_int2_up_packed_bytes(256, 512) == 32 * 1 * 2560
    assert lib.expert_int2_up_packed_bytes(100, 512) == 0
    assert lib.expert_int2_up_packed_bytes(256, 10) == 0


def test_host_argument_checks(so):
    """Rejected before anything is enqueued, so no GPU is needed."""
    from sparse_expert_swiglu_gb300 import _lib
    lib = _lib.lib()
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    assert lib.expert_pack_int2_up(None, 256, 512, fake, None) == -1
    assert lib.expert_pack_int2_up(fake, 100, 512, fake, None) == -2
    assert lib.expert_pack_int2_up(odd, 256, 512, fake, None) == -3
    assert lib.moe_route_topk(fake, 1, 256, fake, 8, 9, 1, fake, fake, None, fake, 1 << 20, None) == -1
    assert lib.moe_route_topk(fake, 1, 300, fake, 8, 2, 1, fake, fake, None, fake, 1 << 20, None) == -2
    assert lib.moe_route_topk(fake, 0, 256, fake, 8, 2, 1, fake, fake, None, fake, 1 << 20, None) == 0
    # the static-scratch router: more than 2048 (token, expert) pairs is refused up front
    assert lib.moe_route_topk_noalloc(fake, 1024, 256, fake, 8, 4, 1, fake, fake, None, None) == -4
    assert lib.moe_route_topk_noalloc(fake, 1, 256, fake, 8, 9, 1, fake, fake, None, None) == -1
    assert lib.moe_route_topk_noalloc(fake, 0, 256, fake, 8, 2, 1, fake, fake, None, None) == 0

    ex = _lib._Experts(8, 4096, 14336, 0x10000, 0x20000, 0x30000, 0x40000)
    layer = _lib._Layer(2, 1, 0x50000, ex, _lib._Experts(0, 4096, 14336, None, None, None, None))
    # B = 0 is a no-op
    assert lib.moe_layer_decode(fake, 0, ctypes.byref(layer), fake, 0, None, fake, 0, None) == 0
    bad = _lib._Layer(9, 1, 0x50000, ex, _lib._Experts(0, 4096, 14336, None, None, None, None))
    assert lib.moe_layer_decode(fake, 1, ctypes.byref(bad), fake, 0, None, fake, 0, None) == -1
    ex_bad_d = _lib._Experts(8, 4000, 14336, 0x10000, 0x20000, 0x30000, 0x40000)
    bad_d = _lib._Layer(2, 1, 0x50000, ex_bad_d, _lib._Experts(0, 4000, 14336, None, None, None, None))
    assert lib.moe_layer_decode(fake, 1, ctypes.byref(bad_d), fake, 0, None, fake, 0, None) == -2
    ex_odd = _lib._Experts(8, 4096, 14336, 0x10008, 0x20000, 0x30000, 0x40000)
    bad_a = _lib._Layer(2, 1, 0x50000, ex_odd, _lib._Experts(0, 4096, 14336, None, None, None, None))
    assert lib.moe_layer_decode(fake, 1, ctypes.byref(bad_a), fake, 0, None, fake, 0, None) == -3
    assert lib.moe_expert_sparse_swiglu(fake, 1, ctypes.byref(ex), 8, fake, None, fake, 0, None) == -1
    # the host-rows layer call: the same checks, before any pointer is looked up
    assert lib.moe_layer_decode_host_rows(fake, 0, ctypes.byref(layer), fake, 0, None, fake, 0, None) == 0
    assert lib.moe_layer_decode_host_rows(fake, 1, ctypes.byref(bad), fake, 0, None, fake, 0, None) == -1
    assert lib.moe_layer_decode_host_rows(fake, 1, ctypes.byref(bad_d), fake, 0, None, fake, 0, None) == -2
    assert lib.moe_layer_decode_host_rows(fake, 1, ctypes.byref(bad_a), fake, 0, None, fake, 0, None) == -3
    assert lib.moe_layer_decode_host_rows(fake, 1, None, fake, 0, None, fake, 0, None) == -1
    assert lib.moe_layer_host_rows_workspace_bytes(ctypes.byref(bad), 1) == 0
    # the expert prefetch hook: argument errors before any CUDA call; nothing to do is OK
    pf = lib.moe_prefetch_experts
    assert pf(None, fake, 4, 0, None) == -1
    assert pf(ctypes.byref(ex), fake, -1, 0, None) == -1
    assert pf(ctypes.byref(ex), fake, 1025, 0, None) == -2
    assert pf(ctypes.byref(ex_bad_d), fake, 4, 0, None) == -2
    assert pf(ctypes.byref(ex_odd), fake, 4, 0, None) == -3
    assert pf(ctypes.byref(ex), None, 4, 0, None) == -1
    assert pf(ctypes.byref(ex), ctypes.c_void_p(0x10002), 4, 0, None) == -3
    assert pf(ctypes.byref(_lib._Experts(0, 4096, 14336, 0x10000, None, None, None)), fake, 4, 0, None) == -2
    assert pf(ctypes.byref(_lib._Experts(8, 4096, 14336, None, None, None, None)), fake, 4, 0, None) == -1
    assert pf(ctypes.byref(ex), None, 0, 0, None) == 0
    # a byte cap below one expert's packed up projection leaves nothing to prefetch
    assert pf(ctypes.byref(ex), fake, 4, lib.expert_int2_up_packed_bytes(4096, 14336) - 1, None) == 0
    # the timeout diagnostic: refused before anything is enqueued
    assert lib.moe_selftest_wait_timeout(None, 1 << 20, 10, None) == -1
    assert lib.moe_selftest_wait_timeout(fake, 1 << 20, 0, None) == -1
    assert lib.moe_selftest_wait_timeout(fake, 4, 10, None) == -4
    assert lib.moe_selftest_wait_timeout(odd, 1 << 20, 10, None) == -3


def test_binding_refuses_host_memory_outside_the_host_rows_call():
    """The binding hands only CUDA tensors to the device path; gate/down rows in host
    memory must be page-locked and go through layer_decode_host_rows (no GPU needed:
    the checks run before any call into the library)."""
    import torch
    from sparse_expert_swiglu_gb300 import _lib
    t = torch.zeros(4)
    with pytest.raises(TypeError, match="CUDA tensor"):
        _lib._need(t, torch.float32, "x")
    with pytest.raises(TypeError, match="page-locked"):
        _lib._need(t, torch.float32, "x", host_ok=True)  # pageable host memory
    ex = _lib.Experts(torch.zeros(1, 8, dtype=torch.uint8), torch.zeros(1, 16, 256, dtype=torch.float16),
                      torch.zeros(1, 16, 256, dtype=torch.float16), torch.zeros(1))
    assert ex.rows_on_host
    with pytest.raises(TypeError):
        ex.c_struct()
    layer = _lib.Layer(torch.zeros(256, 1, dtype=torch.float16), ex, 1)
    with pytest.raises(ValueError, match="layer_decode_host_rows"):
        _lib.layer_decode(torch.zeros(1, 256, dtype=torch.float16), layer)
