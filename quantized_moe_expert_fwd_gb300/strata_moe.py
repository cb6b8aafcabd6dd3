"""Thin Python binding of the C ABI in include/strata_moe.h.

Argument marshalling only: torch CUDA tensors become device pointers, the
current torch stream becomes the call's stream, and a non-OK status raises
StrataError.  Every step of the computation runs in libstrata_moe.so; there
is no fallback, so a missing or unloadable library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

STRATA_OK, STRATA_EINVAL, STRATA_ECUDA, STRATA_EUNSUPPORTED, STRATA_ETIMEOUT, \
    STRATA_EBADROUTE, STRATA_ERANGE = range(7)

_lock = threading.Lock()
_lib = None


class StrataError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == STRATA_ECUDA:
            detail = f" [{load().strata_last_cuda_error().decode()}]"
        super().__init__(f"{fn}: {strata_status_str(status)} ({status}){detail}")


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("group", ctypes.c_int32)]


_LAYER_FIELDS = ("router", "router_bias", "gu_q", "gu_s", "dn_q", "dn_s",
                 "sh_gu_q", "sh_gu_s", "sh_dn_q", "sh_dn_s")


class LayerPtrs(ctypes.Structure):
    _fields_ = [(n + "_dev", ctypes.c_void_p) for n in _LAYER_FIELDS]


_path_override = None


def lib_path() -> str:
    return _path_override or _build.LIB_PATH


def use_library(path: str) -> None:
    """Load `path` instead of libstrata_moe.so (the phase-traced build of the
    same sources); only before the first call loads a library."""
    global _path_override
    with _lock:
        if _lib is not None and path != lib_path():
            raise RuntimeError("a library is already loaded in this process")
        _path_override = path


def load() -> ctypes.CDLL:
    """Load libstrata_moe.so (built in-tree by build.build()); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run quantized_moe_expert_fwd_gb300.build.build()"
                               " (the CUDA library is required; there is no fallback)")
        lib = ctypes.CDLL(path)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        D, L = ctypes.POINTER(Dims), ctypes.POINTER(LayerPtrs)
        sigs = {
            "moe_workspace_bytes": (SZ, [D, I32]),
            "moe_decode_max_tokens": (I32, []),
            "moe_layer_decode_max_tokens": (I32, []),
            "moe_rmsnorm": (I32, [P, I32, I32, ctypes.c_float, P, P]),
            "moe_route": (I32, [D, L, P, I32, P, P, P, P, P, SZ, P]),
            "moe_permute": (I32, [D, P, I32, P, P, P, P, P, SZ, P]),
            "moe_expert_gate_up": (I32, [D, L, P, I32, P, P, P, P, SZ, P]),
            "moe_expert_down": (I32, [D, L, P, I32, P, P, P, SZ, P]),
            "moe_expert_ffn": (I32, [D, L, P, I32, P, P, P, P, SZ, P]),
            "moe_combine": (I32, [D, L, P, I32, P, P, P, P, P, P, SZ, P]),
            "moe_layer_forward": (I32, [D, L, P, I32, P, P, P, P, P, SZ, P]),
            "moe_layer_forward_routed": (I32, [D, L, P, I32, P, P, P, P, SZ, P]),
            "moe_layer_forward_tail_skip": (I32, [D, L, P, I32, I32, P, P, P, P, P, P, P, SZ, P]),
            "moe_block_forward": (I32, [D, L, P, I32, ctypes.c_float, P, P, P, P, P, SZ, P]),
            "moe_stack_forward": (I32, [D, L, I32, P, I32, ctypes.c_float, P, P, P, P, SZ, P]),
            "moe_decode_route": (I32, [D, L, P, I32, I32, P, SZ, P]),
            "moe_decode_gate_up": (I32, [D, L, P, I32, P, P, P, P, P, P, SZ, P]),
            "moe_decode_down_combine": (I32, [D, L, I32, P, P, P, SZ, P]),
            "moe_layer_forward_static": (I32, [D, L, P, I32, P, P, P, P, P]),
            "moe_layer_profile": (I32, [D, L, P, I32, P, P, SZ, P, P, I32, P]),
            "moe_layer_path": (I32, [D, I32, I32]),
            "moe_layer_bucketing": (I32, [D, I32, P, SZ, P, P, P, P, P]),
            "moe_get_device_status": (I32, [P, P]),
            "strata_set_grid_wait_limit": (None, [ctypes.c_uint32]),
            "strata_px_trace_read": (I32, [P, SZ]),
            "strata_status_str": (ctypes.c_char_p, [I32]),
            "strata_last_cuda_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


EXPORTED = ("moe_workspace_bytes", "moe_decode_max_tokens", "moe_layer_decode_max_tokens",
            "moe_rmsnorm", "moe_route",
            "moe_permute", "moe_expert_gate_up", "moe_expert_down", "moe_expert_ffn",
            "moe_combine", "moe_layer_forward", "moe_layer_forward_routed",
            "moe_layer_forward_tail_skip",
            "moe_block_forward", "moe_stack_forward", "moe_decode_route", "moe_decode_gate_up",
            "moe_decode_down_combine", "moe_layer_forward_static", "moe_layer_profile",
            "moe_layer_path", "moe_layer_bucketing", "moe_get_device_status",
            "strata_set_grid_wait_limit", "strata_px_trace_read",
            "strata_status_str", "strata_last_cuda_error")


# ---------------------------------------------------------------- helpers
def dims_struct(d) -> Dims:
    return Dims(int(d.hidden), int(d.n_experts), int(d.top_k), int(d.inter),
                int(d.shared_inter), int(getattr(d, "group", 32)))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_contiguous():
        raise ValueError("tensors passed to strata_moe must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != STRATA_OK:
        raise StrataError(fn, status)


def strata_status_str(status: int) -> str:
    return load().strata_status_str(int(status)).decode()


class DeviceLayer:
    """One layer's packed planes resident on the GPU (torch tensors keep the
    memory alive) plus the pointer struct the ABI takes."""

    def __init__(self, planes: dict, device="cuda"):
        self.tensors = {}
        for n in _LAYER_FIELDS:
            a = planes.get(n)
            if a is None:
                self.tensors[n] = None
                continue
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                t = torch.from_numpy(a.view(np.int16)).to(device)
            else:
                t = torch.from_numpy(a).to(device)
            self.tensors[n] = t
        self.ptrs = LayerPtrs(*[(None if self.tensors[n] is None else self.tensors[n].data_ptr())
                                for n in _LAYER_FIELDS])

    def with_bias(self, bias, device="cuda") -> "DeviceLayer":
        """The same resident planes with another router bias (fp32 [E] array,
        or None): no plane is copied again."""
        other = DeviceLayer.__new__(DeviceLayer)
        other.tensors = dict(self.tensors)
        other.tensors["router_bias"] = (None if bias is None else
                                        torch.from_numpy(np.ascontiguousarray(bias, dtype=np.float32))
                                        .to(device))
        other.ptrs = LayerPtrs(*[(None if other.tensors[n] is None else other.tensors[n].data_ptr())
                                 for n in _LAYER_FIELDS])
        return other

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors.values() if t is not None)


def make_workspace(dims, max_tokens: int, device="cuda") -> torch.Tensor:
    n = moe_workspace_bytes(dims, max_tokens)
    if n == 0:
        raise StrataError("moe_workspace_bytes", STRATA_EINVAL)
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ------------------------------------------------------------ ABI mirrors
def moe_workspace_bytes(dims, max_tokens: int) -> int:
    d = dims_struct(dims)
    return int(load().moe_workspace_bytes(ctypes.byref(d), int(max_tokens)))


def moe_decode_max_tokens() -> int:
    return int(load().moe_decode_max_tokens())


def moe_layer_decode_max_tokens() -> int:
    return int(load().moe_layer_decode_max_tokens())


def moe_rmsnorm(r, x, eps: float = 1e-6, stream=None):
    T, H = r.shape
    _check("moe_rmsnorm", load().moe_rmsnorm(_ptr(r), T, H, ctypes.c_float(eps), _ptr(x),
                                             _stream(stream)))


def moe_route(dims, layer: DeviceLayer, x, ids, weights, shared_gate, ws, logits=None,
              stream=None):
    d = dims_struct(dims)
    _check("moe_route", load().moe_route(ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x),
                                         x.shape[0], _ptr(ids), _ptr(weights),
                                         _ptr(shared_gate), _ptr(logits), _ptr(ws),
                                         ws.numel(), _stream(stream)))


def moe_permute(dims, ids, counts, offsets, perm, inv_perm, ws, stream=None):
    d = dims_struct(dims)
    _check("moe_permute", load().moe_permute(ctypes.byref(d), _ptr(ids), ids.shape[0],
                                             _ptr(counts), _ptr(offsets), _ptr(perm),
                                             _ptr(inv_perm), _ptr(ws), ws.numel(),
                                             _stream(stream)))


def moe_expert_gate_up(dims, layer: DeviceLayer, x, offsets, perm, h, ws, stream=None):
    d = dims_struct(dims)
    _check("moe_expert_gate_up", load().moe_expert_gate_up(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(offsets),
        _ptr(perm), _ptr(h), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_down(dims, layer: DeviceLayer, h, T: int, offsets, y, ws, stream=None):
    d = dims_struct(dims)
    _check("moe_expert_down", load().moe_expert_down(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(h), int(T), _ptr(offsets), _ptr(y),
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_ffn(dims, layer: DeviceLayer, x, offsets, perm, y, ws, stream=None):
    d = dims_struct(dims)
    _check("moe_expert_ffn", load().moe_expert_ffn(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(offsets),
        _ptr(perm), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


def moe_combine(dims, layer: DeviceLayer, x, y, inv_perm, weights, shared_gate, out, ws,
                stream=None):
    d = dims_struct(dims)
    _check("moe_combine", load().moe_combine(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(y),
        _ptr(inv_perm), _ptr(weights), _ptr(shared_gate), _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_layer_forward(dims, layer: DeviceLayer, x, out, ws, ids=None, weights=None,
                      shared_gate=None, stream=None):
    d = dims_struct(dims)
    _check("moe_layer_forward", load().moe_layer_forward(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(ids),
        _ptr(weights), _ptr(shared_gate), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_forward_routed(dims, layer: DeviceLayer, x, ids, weights, out, ws, stream=None):
    d = dims_struct(dims)
    _check("moe_layer_forward_routed", load().moe_layer_forward_routed(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(ids),
        _ptr(weights), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_layer_forward_tail_skip(dims, layer: DeviceLayer, x, out, ws, tail_skip: int,
                                forced_ids=None, forced_weights=None, ids=None, weights=None,
                                shared_gate=None, stream=None):
    d = dims_struct(dims)
    _check("moe_layer_forward_tail_skip", load().moe_layer_forward_tail_skip(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], int(tail_skip),
        _ptr(forced_ids), _ptr(forced_weights), _ptr(ids), _ptr(weights), _ptr(shared_gate),
        _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_block_forward(dims, layer: DeviceLayer, resid, ws, eps: float = 1e-6, ids=None,
                      weights=None, x_out=None, out=None, stream=None):
    d = dims_struct(dims)
    _check("moe_block_forward", load().moe_block_forward(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(resid), resid.shape[0],
        ctypes.c_float(eps), _ptr(ids), _ptr(weights), _ptr(x_out), _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_stack_forward(dims, layers, resid, ws, eps: float = 1e-6, ids=None, weights=None,
                      out=None, stream=None):
    """resid (fp32 [T][H], in/out) through every layer of `layers` (DeviceLayer
    list): x = bf16(rmsnorm(resid)); resid += layer(x).  ids / weights:
    optional [n_layers][T][K] forced routing."""
    d = dims_struct(dims)
    arr = (LayerPtrs * len(layers))(*[dl.ptrs for dl in layers])
    _check("moe_stack_forward", load().moe_stack_forward(
        ctypes.byref(d), arr, len(layers), _ptr(resid), resid.shape[0], ctypes.c_float(eps),
        _ptr(ids), _ptr(weights), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_decode_route(dims, layer: DeviceLayer, x, ws, forced: bool = False, stream=None):
    d = dims_struct(dims)
    _check("moe_decode_route", load().moe_decode_route(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], int(bool(forced)),
        _ptr(ws), ws.numel(), _stream(stream)))


def moe_decode_gate_up(dims, layer: DeviceLayer, x, ws, forced_ids=None, forced_weights=None,
                       ids=None, weights=None, shared_gate=None, stream=None):
    d = dims_struct(dims)
    _check("moe_decode_gate_up", load().moe_decode_gate_up(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(forced_ids),
        _ptr(forced_weights), _ptr(ids), _ptr(weights), _ptr(shared_gate), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_decode_down_combine(dims, layer: DeviceLayer, T: int, out, ws, resid=None, stream=None):
    d = dims_struct(dims)
    _check("moe_decode_down_combine", load().moe_decode_down_combine(
        ctypes.byref(d), ctypes.byref(layer.ptrs), int(T), _ptr(out), _ptr(resid), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_layer_forward_static(dims, layer: DeviceLayer, x, out, ids=None, weights=None,
                             shared_gate=None, stream=None):
    """moe_layer_forward on the library's own fixed workspace (no caller
    allocation); see include/strata_moe.h for its limits."""
    d = dims_struct(dims)
    _check("moe_layer_forward_static", load().moe_layer_forward_static(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(ids),
        _ptr(weights), _ptr(shared_gate), _ptr(out), _stream(stream)))


PROFILE_PERSISTENT = ("k_persist",)
PROFILE_DECODE = ("k_route", "k_gate_up", "k_down")
PROFILE_PREFILL = ("router_gemm", "select", "count", "scan", "scatter", "gather",
                   "gemm_gate_up", "gemm_down", "combine")
# the tcgen05 path at T <= 32: the bucketing is one kernel
PROFILE_PREFILL_SMALL = ("router_gemm", "select", "bucket", "gather", "gemm_gate_up",
                         "gemm_down", "combine")


def moe_layer_profile(dims, layer: DeviceLayer, x, out, ws, stream=None):
    """Per-kernel durations (microseconds, launch order) of one layer forward."""
    d = dims_struct(dims)
    us = (ctypes.c_float * 64)()
    n = ctypes.c_int32(0)
    _check("moe_layer_profile", load().moe_layer_profile(
        ctypes.byref(d), ctypes.byref(layer.ptrs), _ptr(x), x.shape[0], _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream), us, 64, ctypes.byref(n)))
    # which kernels ran: the persistent path launches one, the decode path
    # three, the tensor-core path seven (T <= 32) or nine
    names = {len(PROFILE_PERSISTENT): PROFILE_PERSISTENT, len(PROFILE_DECODE): PROFILE_DECODE,
             len(PROFILE_PREFILL_SMALL): PROFILE_PREFILL_SMALL}.get(n.value, PROFILE_PREFILL)
    return {names[i] if i < len(names) else f"k{i}": float(us[i]) for i in range(n.value)}


PATH_PERSISTENT, PATH_DECODE, PATH_TC = 1, 2, 3


def moe_layer_path(dims, T: int, forced: bool = False) -> int:
    """Which kernels a whole-layer call of T tokens runs (PATH_*; 0: none)."""
    d = dims_struct(dims)
    return int(load().moe_layer_path(ctypes.byref(d), int(T), 1 if forced else 0))


def moe_layer_bucketing(dims, T: int, ws, counts, offsets, perm, inv, stream=None):
    """The bucketing the last whole-layer call on `ws` made (int32 tensors)."""
    d = dims_struct(dims)
    _check("moe_layer_bucketing", load().moe_layer_bucketing(
        ctypes.byref(d), int(T), _ptr(ws), ws.numel(), _ptr(counts), _ptr(offsets), _ptr(perm),
        _ptr(inv), _stream(stream)))


def strata_px_trace_read(nbytes: int = 1024 * 4 * 16 * 8):
    """The persistent kernel's phase timestamps of its last launch, as a
    numpy uint64 array [CTA][slot][point] (a library built with
    build.build(trace=True) only; points and slots as in strata_moe.h)."""
    buf = np.zeros(nbytes // 8, dtype=np.uint64)
    _check("strata_px_trace_read", load().strata_px_trace_read(buf.ctypes.data, buf.nbytes))
    return buf.reshape(-1, 4, 16)


def strata_set_grid_wait_limit(polls: int) -> None:
    """Testing hook: polls before a persistent-kernel grid barrier gives up
    (0: the default)."""
    load().strata_set_grid_wait_limit(int(polls))


def moe_get_device_status(ws, stream=None) -> int:
    return int(load().moe_get_device_status(_ptr(ws), _stream(stream)))
