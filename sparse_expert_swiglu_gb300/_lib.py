"""ctypes binding of the C ABI in include/sparse_expert_swiglu.h.

Argument marshalling only: every step of the MoE path runs in the CUDA library.
torch provides device memory and the current stream.  There is no fallback: if
the library is missing, `lib()` raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import build as _build

MOE_OK = 0
_STATUS = {
    0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "misaligned pointer",
    -4: "workspace too small", -5: "CUDA error", -6: "device-side wait timed out",
    -7: "out of memory",
}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({status})")
        self.status = status


class _Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("up_packed", ctypes.c_void_p), ("gate_t", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("thr", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int32), ("renorm", ctypes.c_int32), ("w_router", ctypes.c_void_p),
                ("routed", _Experts), ("shared", _Experts)]


class _Debug(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("mask", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("events", ctypes.POINTER(ctypes.c_void_p))]


_LIB = None
_SIGS = {
    "expert_int2_up_packed_bytes": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32]),
    "expert_pack_int2_up": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    "expert_unpack_int2_up": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p]),
    "moe_route_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 3),
    "moe_route_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p]),
    "moe_route_topk_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "moe_expert_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 3),
    "moe_expert_sparse_swiglu": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32,
                                                ctypes.POINTER(_Experts), ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.POINTER(_Debug),
                                                ctypes.c_void_p, ctypes.c_size_t,
                                                ctypes.c_void_p]),
    "moe_layer_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(_Layer), ctypes.c_int32]),
    "moe_layer_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Layer),
                                        ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Debug),
                                        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_layer_path": (ctypes.c_int32, [ctypes.POINTER(_Layer), ctypes.c_int32]),
    "moe_layer_host_rows_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(_Layer), ctypes.c_int32]),
    "moe_layer_decode_host_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Layer),
                                                  ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Debug),
                                                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_prefetch_experts": (ctypes.c_int, [ctypes.POINTER(_Experts), ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_size_t, ctypes.c_void_p]),
    "moe_eam_add_counts": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_void_p]),
    "moe_eamc_bytes": (ctypes.c_size_t, [ctypes.c_int32] * 3),
    "moe_eamc_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_int32]),
    "moe_eamc_insert": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_eamc_size": (ctypes.c_int32, [ctypes.c_void_p]),
    "moe_eamc_entry": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "moe_eamc_match": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "moe_eamc_predict": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p]),
    "moe_expert_cache_bytes": (ctypes.c_size_t, [ctypes.c_int32]),
    "moe_expert_cache_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32]),
    "moe_expert_cache_lookup": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p,
                                               ctypes.c_void_p]),
    "moe_expert_cache_contents": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32,
                                                 ctypes.c_void_p]),
    "moe_get_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}
EXPORTED = tuple(_SIGS)


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path}); run __graft_entry__.build()")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status)


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, host_ok: bool = False) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor" + (" or page-locked host tensor" if host_ok else ""))
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---------------------------------------------------------------------------
# workspace
# ---------------------------------------------------------------------------

class Workspace:
    """A zero-initialised device workspace (256-byte aligned torch allocation)."""

    def __init__(self, nbytes: int, device=None):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device or "cuda")
        _check("moe_workspace_init", lib().moe_workspace_init(_ptr(self.buf), self.buf.numel(), _stream()))

    def ptr(self):
        return _ptr(self.buf)

    def status(self) -> int:
        """Synchronise and return (and clear) the first device-side error."""
        return lib().moe_get_status(self.ptr(), _stream())


# ---------------------------------------------------------------------------
# INT2 up projection
# ---------------------------------------------------------------------------

def packed_bytes(d: int, f: int) -> int:
    return int(lib().expert_int2_up_packed_bytes(d, f))


def pack_int2_up(w_up: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """W^up fp16 [d, f] -> packed INT2 bytes (uint8 [packed_bytes(d, f)])."""
    _need(w_up, torch.float16, "w_up")
    d, f = w_up.shape
    if out is None:
        out = torch.empty(packed_bytes(d, f), dtype=torch.uint8, device=w_up.device)
    _check("expert_pack_int2_up", lib().expert_pack_int2_up(_ptr(w_up), d, f, _ptr(out), _stream()))
    return out


def unpack_int2_up(packed: torch.Tensor, d: int, f: int):
    """Packed bytes -> (q uint8 [d, f], scale fp16 [d/64, f], zero fp16 [d/64, f])."""
    _need(packed, torch.uint8, "packed")
    q = torch.empty((d, f), dtype=torch.uint8, device=packed.device)
    s = torch.empty((d // 64, f), dtype=torch.float16, device=packed.device)
    z = torch.empty((d // 64, f), dtype=torch.float16, device=packed.device)
    _check("expert_unpack_int2_up",
           lib().expert_unpack_int2_up(_ptr(packed), d, f, _ptr(q), _ptr(s), _ptr(z), _stream()))
    return q, s, z


# ---------------------------------------------------------------------------
# experts and layers
# ---------------------------------------------------------------------------

@dataclass
class Experts:
    """A stack of E equally shaped experts (device tensors).

    up_packed uint8 [E, packed_bytes(d, f)]; gate_t fp16 [E, f, d] (row i = column i
    of W^gate); down fp16 [E, f, d] (row i = row i of W^down); thr fp32 [E]."""
    up_packed: torch.Tensor
    gate_t: torch.Tensor
    down: torch.Tensor
    thr: torch.Tensor

    @property
    def E(self):
        return self.gate_t.shape[0]

    @property
    def f(self):
        return self.gate_t.shape[1]

    @property
    def d(self):
        return self.gate_t.shape[2]

    @property
    def interleaved(self) -> bool:
        """gate and down rows share one buffer [E, f, 2, d] (gate row i, then down row i)."""
        return (self.gate_t.dim() == 3 and self.gate_t.stride() == self.down.stride()
                and self.gate_t.stride(1) == 2 * self.d
                and self.down.data_ptr() == self.gate_t.data_ptr() + 2 * self.d)

    @property
    def rows_on_host(self) -> bool:
        """gate_t and down live in page-locked host memory (see to_host_rows)."""
        return not self.gate_t.is_cuda

    def c_struct(self, host_rows: bool = False) -> _Experts:
        """The C description; host_rows=True admits gate_t/down in page-locked host memory
        (only moe_layer_decode_host_rows reads such rows)."""
        _need(self.up_packed, torch.uint8, "up_packed")
        _need(self.thr, torch.float32, "thr")
        if self.interleaved:
            both = self.gate_t.as_strided((self.E, self.f, 2, self.d),
                                          (self.f * 2 * self.d, 2 * self.d, self.d, 1))
            _need(both, torch.float16, "gate_t/down (interleaved)", host_rows)
        else:
            _need(self.gate_t, torch.float16, "gate_t", host_rows)
            _need(self.down, torch.float16, "down", host_rows)
        return _Experts(self.E, self.d, self.f, self.up_packed.data_ptr(), self.gate_t.data_ptr(),
                        self.down.data_ptr(), self.thr.data_ptr())

    def to_host_rows(self) -> "Experts":
        """A copy whose gate and down rows live in page-locked host memory (interleaving
        kept); the packed up projection and the thresholds stay where they are."""
        if self.interleaved:
            both = self.gate_t.as_strided((self.E, self.f, 2, self.d),
                                          (self.f * 2 * self.d, 2 * self.d, self.d, 1))
            h = both.cpu().pin_memory()
            return Experts(self.up_packed, h[:, :, 0, :], h[:, :, 1, :], self.thr)
        return Experts(self.up_packed, self.gate_t.cpu().pin_memory(), self.down.cpu().pin_memory(), self.thr)

    @staticmethod
    def from_dense(w_up: torch.Tensor, gate_t: torch.Tensor, down: torch.Tensor,
                   thr: torch.Tensor, interleave: bool = False) -> "Experts":
        """Pack every W^up [E, d, f] with the library's INT2 quantiser.  interleave=True
        stores gate and down rows in one buffer [E, f, 2, d], so that a kept column's two
        rows are one contiguous 4d-byte read."""
        E, d, f = w_up.shape
        up = torch.empty((E, packed_bytes(d, f)), dtype=torch.uint8, device=w_up.device)
        for e in range(E):
            pack_int2_up(w_up[e].contiguous(), up[e])
        if interleave:
            gd = torch.empty((E, f, 2, d), dtype=gate_t.dtype, device=gate_t.device)
            gd[:, :, 0, :] = gate_t
            gd[:, :, 1, :] = down
            return Experts(up, gd[:, :, 0, :], gd[:, :, 1, :], thr.contiguous())
        return Experts(up, gate_t.contiguous(), down.contiguous(), thr.contiguous())


def _empty_experts(d: int, f: int) -> _Experts:
    return _Experts(0, d, f, None, None, None, None)


@dataclass
class Layer:
    w_router: torch.Tensor       # fp16 [d, E]
    routed: Experts
    k: int
    renorm: bool = True
    shared: Optional[Experts] = None

    def c_struct(self, host_rows: bool = False) -> _Layer:
        _need(self.w_router, torch.float16, "w_router")
        r = self.routed.c_struct(host_rows)
        s = self.shared.c_struct(host_rows) if self.shared is not None else _empty_experts(r.d, r.f)
        return _Layer(self.k, 1 if self.renorm else 0, self.w_router.data_ptr(), r, s)

    @property
    def n_slots(self) -> int:
        return self.k + (self.shared.E if self.shared is not None else 0)


def _debug(B: int, S: int, f: int, k: int, device, with_route: bool):
    t = dict(mask=torch.zeros((B, S, (f + 31) // 32), dtype=torch.int32, device=device),
             v=torch.zeros((B, S, f), dtype=torch.float32, device=device))
    if with_route:
        t["topk_idx"] = torch.zeros((B, k), dtype=torch.int32, device=device)
        t["topk_w"] = torch.zeros((B, k), dtype=torch.float32, device=device)
    dbg = _Debug(_ptr(t.get("topk_idx")), _ptr(t.get("topk_w")), _ptr(t["mask"]), _ptr(t["v"]), None)
    return dbg, t


def _with_events(dbg, events):
    """Attach 5 timing events (torch.cuda.Event(enable_timing=True)) to a debug block."""
    if events is None:
        return dbg
    if len(events) != 5:
        raise ValueError("need 5 events")
    for ev in events:
        if ev.cuda_event == 0:  # torch creates the event on its first record
            ev.record()
    arr = (ctypes.c_void_p * 5)(*[ev.cuda_event for ev in events])
    if dbg is None:
        dbg = _Debug(None, None, None, None, None)
    dbg.events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    dbg._keep = arr
    return dbg


def route_workspace_bytes(B: int, E: int, k: int) -> int:
    return int(lib().moe_route_workspace_bytes(B, E, k))


def route_topk(x: torch.Tensor, w_router: torch.Tensor, k: int, renorm: bool = True,
               ws: Optional[Workspace] = None):
    """-> (topk_idx int32 [B, k], topk_w fp32 [B, k], expert_count int32 [E])."""
    _need(x, torch.float16, "x")
    _need(w_router, torch.float16, "w_router")
    B, d = x.shape
    E = w_router.shape[1]
    if ws is None:
        ws = Workspace(route_workspace_bytes(B, E, k), x.device)
    idx = torch.empty((B, k), dtype=torch.int32, device=x.device)
    w = torch.empty((B, k), dtype=torch.float32, device=x.device)
    cnt = torch.empty((E,), dtype=torch.int32, device=x.device)
    _check("moe_route_topk", lib().moe_route_topk(_ptr(x), B, d, _ptr(w_router), E, k,
                                                  1 if renorm else 0, _ptr(idx), _ptr(w),
                                                  _ptr(cnt), ws.ptr(), ws.nbytes, _stream()))
    return idx, w, cnt


ROUTE_NOALLOC_MAX_PAIRS = 2048


def route_topk_noalloc(x: torch.Tensor, w_router: torch.Tensor, k: int, renorm: bool = True):
    """route_topk through the entry point that uses the library's static scratch
    instead of a workspace (B * k <= ROUTE_NOALLOC_MAX_PAIRS)."""
    _need(x, torch.float16, "x")
    _need(w_router, torch.float16, "w_router")
    B, d = x.shape
    E = w_router.shape[1]
    idx = torch.empty((B, k), dtype=torch.int32, device=x.device)
    w = torch.empty((B, k), dtype=torch.float32, device=x.device)
    cnt = torch.empty((E,), dtype=torch.int32, device=x.device)
    _check("moe_route_topk_noalloc",
           lib().moe_route_topk_noalloc(_ptr(x), B, d, _ptr(w_router), E, k,
                                        1 if renorm else 0, _ptr(idx), _ptr(w), _ptr(cnt),
                                        _stream()))
    return idx, w, cnt


def expert_workspace_bytes(n: int, d: int, f: int) -> int:
    return int(lib().moe_expert_workspace_bytes(n, d, f))


def expert_sparse_swiglu(x: torch.Tensor, experts: Experts, expert: int,
                         ws: Optional[Workspace] = None, debug: bool = False,
                         out: Optional[torch.Tensor] = None, events=None,
                         c_experts: Optional[_Experts] = None):
    """One sparse SwiGLU expert on every row of x (fp16 [n, d]) -> y fp16 [n, d]
    (and, with debug, a dict with mask int32 [n, 1, ceil(f/32)] and v fp32 [n, 1, f])."""
    _need(x, torch.float16, "x")
    n, d = x.shape
    ex = c_experts if c_experts is not None else experts.c_struct()
    if ws is None:
        ws = Workspace(expert_workspace_bytes(n, d, experts.f), x.device)
    y = out if out is not None else torch.empty_like(x)
    dbg, dt = (None, None)
    if debug:
        dbg, dt = _debug(n, 1, experts.f, 1, x.device, False)
    dbg = _with_events(dbg, events)
    _check("moe_expert_sparse_swiglu",
           lib().moe_expert_sparse_swiglu(_ptr(x), n, ctypes.byref(ex), expert, _ptr(y),
                                          ctypes.byref(dbg) if dbg is not None else None,
                                          ws.ptr(), ws.nbytes, _stream()))
    return (y, dt) if debug else y


def layer_workspace_bytes(layer: Layer, B: int) -> int:
    c = layer.c_struct()
    return int(lib().moe_layer_workspace_bytes(ctypes.byref(c), B))


def layer_path(layer: Layer, B: int) -> str:
    """Which kernels layer_decode runs: 'decode_fused' (one token, d <= 4096: one kernel),
    'decode' (two tokens, or one token with 4096 < d <= 6144: an up kernel and a gather
    kernel), 'batched' (16 to 64 tokens, d <= 4096, at least 6 tokens per routed expert
    on average: router, up kernel, then per-expert kept-row lists and gate and down passes
    that read each kept row once per expert), 'decode_pairs' (three to six tokens of a
    shape the decode path takes, three or four with more than 16 routed experts: two at
    a time through it) or
    'general' (router, up, gather and combine kernels)."""
    r = int(lib().moe_layer_path(ctypes.byref(layer.c_struct()), B))
    if r < 0:
        raise MoeError("moe_layer_path", r)
    return {1: "decode", 2: "decode_fused", 3: "batched", 4: "decode_pairs"}.get(r, "general")


def layer_decode(x: torch.Tensor, layer: Layer, rmsnorm: bool = False,
                 ws: Optional[Workspace] = None, debug: bool = False,
                 out: Optional[torch.Tensor] = None, c_layer: Optional[_Layer] = None,
                 events=None):
    """One MoE decode layer on x fp16 [B, d] -> y fp16 [B, d] (and the debug dict)."""
    if layer.routed.rows_on_host or (layer.shared is not None and layer.shared.rows_on_host):
        raise ValueError("gate/down rows in host memory: use layer_decode_host_rows")
    _need(x, torch.float16, "x")
    B, d = x.shape
    c = c_layer if c_layer is not None else layer.c_struct()
    if ws is None:
        ws = Workspace(int(lib().moe_layer_workspace_bytes(ctypes.byref(c), B)), x.device)
    y = out if out is not None else torch.empty_like(x)
    dbg, dt = (None, None)
    if debug:
        dbg, dt = _debug(B, layer.n_slots, layer.routed.f, layer.k, x.device, True)
    dbg = _with_events(dbg, events)
    _check("moe_layer_decode",
           lib().moe_layer_decode(_ptr(x), B, ctypes.byref(c), _ptr(y), 1 if rmsnorm else 0,
                                  ctypes.byref(dbg) if dbg is not None else None,
                                  ws.ptr(), ws.nbytes, _stream()))
    return (y, dt) if debug else y


def prefetch_experts(experts: Experts, idx: torch.Tensor, max_bytes: int = 0) -> None:
    """L2-prefetch the packed up projections of the experts listed in idx (device int32,
    any shape; repeats and ids outside [0, E) ignored) on the current stream."""
    _need(idx, torch.int32, "idx")
    n = idx.numel()
    _check("moe_prefetch_experts",
           lib().moe_prefetch_experts(ctypes.byref(experts.c_struct()), _ptr(idx) if n else None, n,
                                      max_bytes, _stream()))


def layer_host_rows_workspace_bytes(layer: Layer, B: int) -> int:
    c = layer.c_struct(host_rows=True)
    return int(lib().moe_layer_host_rows_workspace_bytes(ctypes.byref(c), B))


def layer_decode_host_rows(x: torch.Tensor, layer: Layer, rmsnorm: bool = False,
                           ws: Optional[Workspace] = None, debug: bool = False,
                           out: Optional[torch.Tensor] = None, c_layer: Optional[_Layer] = None,
                           events=None):
    """layer_decode with the experts' gate/down rows in page-locked host memory
    (Experts.to_host_rows): only the kept rows cross to the GPU.  One or two tokens."""
    _need(x, torch.float16, "x")
    B, d = x.shape
    c = c_layer if c_layer is not None else layer.c_struct(host_rows=True)
    if ws is None:
        ws = Workspace(int(lib().moe_layer_host_rows_workspace_bytes(ctypes.byref(c), B)), x.device)
    y = out if out is not None else torch.empty_like(x)
    dbg, dt = (None, None)
    if debug:
        dbg, dt = _debug(B, layer.n_slots, layer.routed.f, layer.k, x.device, True)
    dbg = _with_events(dbg, events)
    _check("moe_layer_decode_host_rows",
           lib().moe_layer_decode_host_rows(_ptr(x), B, ctypes.byref(c), _ptr(y), 1 if rmsnorm else 0,
                                            ctypes.byref(dbg) if dbg is not None else None,
                                            ws.ptr(), ws.nbytes, _stream()))
    return (y, dt) if debug else y


# ---------------------------------------------------------------------------
# expert activation tracking and the expert cache (host; numpy-backed buffers)
# ---------------------------------------------------------------------------

def _np_ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a, shape, name: str) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    if a.shape != shape:
        raise ValueError(f"{name} must have shape {shape}, got {a.shape}")
    return a


def eam_add_counts(eam: np.ndarray, layer: int, counts) -> None:
    """eam[layer] += counts (in place; eam int32 [L, E], C-contiguous)."""
    if eam.dtype != np.int32 or not eam.flags.c_contiguous or eam.ndim != 2:
        raise TypeError("eam must be a C-contiguous int32 [L, E] array")
    L, E = eam.shape
    c = _i32(counts, (E,), "counts")
    _check("moe_eam_add_counts", lib().moe_eam_add_counts(_np_ptr(eam), L, E, layer, _np_ptr(c)))


class EAMC:
    """A fixed-capacity collection of request-level expert activation matrices (L x E)."""

    def __init__(self, L: int, E: int, capacity: int):
        self.L, self.E, self.capacity = L, E, capacity
        n = int(lib().moe_eamc_bytes(L, E, capacity))
        if n == 0:
            raise ValueError("invalid EAMC size")
        self._buf = np.zeros(n, dtype=np.uint8)
        _check("moe_eamc_init", lib().moe_eamc_init(_np_ptr(self._buf), n, L, E, capacity))

    def ptr(self):
        return _np_ptr(self._buf)

    def __len__(self) -> int:
        return int(lib().moe_eamc_size(self.ptr()))

    def insert(self, ream) -> int:
        """Append, or replace the nearest stored entry when full; returns the slot."""
        r = _i32(ream, (self.L, self.E), "ream")
        slot = ctypes.c_int32(-1)
        _check("moe_eamc_insert", lib().moe_eamc_insert(self.ptr(), _np_ptr(r), ctypes.byref(slot)))
        return slot.value

    def entry(self, i: int) -> np.ndarray:
        out = np.empty((self.L, self.E), dtype=np.int32)
        _check("moe_eamc_entry", lib().moe_eamc_entry(self.ptr(), i, _np_ptr(out)))
        return out

    def match(self, cur, n_match: int = 1):
        """(indices, cosine distances) of the n_match nearest entries."""
        c = _i32(cur, (self.L, self.E), "cur")
        idx = np.empty(n_match, dtype=np.int32)
        dist = np.empty(n_match, dtype=np.float64)
        nf = ctypes.c_int32(0)
        _check("moe_eamc_match", lib().moe_eamc_match(self.ptr(), _np_ptr(c), n_match, _np_ptr(idx),
                                                      _np_ptr(dist), ctypes.byref(nf)))
        return idx[:nf.value], dist[:nf.value]

    def predict(self, cur, layer: int, n_match: int = 1) -> np.ndarray:
        """PredictEAM: float64 [L, E] activation likelihoods for the current layer."""
        c = _i32(cur, (self.L, self.E), "cur")
        out = np.empty((self.L, self.E), dtype=np.float64)
        _check("moe_eamc_predict", lib().moe_eamc_predict(self.ptr(), _np_ptr(c), layer, n_match, _np_ptr(out)))
        return out


class ExpertCache:
    """The sparsity-aware expert cache (MoE-Infinity's Algorithm 1) over (layer, expert) ids."""

    def __init__(self, capacity: int, L: int, E: int):
        self.capacity, self.L, self.E = capacity, L, E
        n = int(lib().moe_expert_cache_bytes(capacity))
        if n == 0:
            raise ValueError("invalid cache capacity")
        self._buf = np.zeros(n, dtype=np.uint8)
        _check("moe_expert_cache_init", lib().moe_expert_cache_init(_np_ptr(self._buf), n, capacity, L, E))

    def lookup(self, eamc: EAMC, cur, layer: int, expert: int, n_match: int = 1, eps: float = 1e-4):
        """(hit, evicted (layer, expert) or None)."""
        c = _i32(cur, (self.L, self.E), "cur")
        hit = ctypes.c_int32(0)
        ev = np.full(2, -1, dtype=np.int32)
        _check("moe_expert_cache_lookup",
               lib().moe_expert_cache_lookup(_np_ptr(self._buf), eamc.ptr(), _np_ptr(c), layer, expert, n_match,
                                             float(eps), ctypes.byref(hit), _np_ptr(ev)))
        return bool(hit.value), (None if ev[0] < 0 else (int(ev[0]), int(ev[1])))

    def contents(self):
        out = np.empty(2 * self.capacity, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check("moe_expert_cache_contents", lib().moe_expert_cache_contents(_np_ptr(self._buf), _np_ptr(out),
                                                                            ctypes.byref(n)))
        return [(int(out[2 * i]), int(out[2 * i + 1])) for i in range(n.value)]
