"""Python binding of libfp4moe (include/fp4moe.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels.  This module
loads the in-tree shared library, turns torch tensors into device pointers and
the current CUDA stream, and raises on a non-zero status.  There is no CPU or
PyTorch fallback: if the library is missing or was not built, every call fails
loudly (``build()`` compiles it).

With the environment variable FP4MOE_BOUNDS_CHECK=1 set before the first
call, the bounds-checked variant of the library (libfp4moe_checked.so, same
sources, every data-dependent index checked on the device; a failed check
records ERR_BOUNDS) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

__all__ = [
    "FP4MoEError", "ACT_BF16", "ACT_FP8", "W13_GATE_UP", "W13_UP_GATE",
    "FLAG_NO_REQUANT", "FLAG_KEEP_GROUP16", "FLAG_GS_INVERTED", "load", "build", "exported_symbols",
    "requant_fp4_gran_k", "act_quant", "route_debug", "route_workspace_size",
    "prepare_weights", "PackedWeights", "moe_workspace_size", "moe_forward",
    "moe_workspace_size_host", "moe_forward_host", "status_string",
    "last_device_error", "set_stage_events", "STAGE_NAMES",
    "test_wait_timeout", "test_bounds_check", "build_flags", "variant",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, \
    ERR_TIMEOUT, ERR_BOUNDS = range(7)
BUILD_BOUNDS_CHECK = 1
W13_GATE_UP, W13_UP_GATE = 0, 1
ACT_BF16, ACT_FP8 = 0, 1
FLAG_NO_REQUANT = 0x100
FLAG_KEEP_GROUP16 = 0x200
FLAG_GS_INVERTED = 0x400

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(
    __file__))), "include", "fp4moe.h")
_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class FP4MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class PackedDesc(ctypes.Structure):
    _fields_ = [
        ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("I", ctypes.c_int32),
        ("gran_k", ctypes.c_int32), ("act_mode", ctypes.c_int32),
        ("w13_layout", ctypes.c_int32), ("k_tile", ctypes.c_int32),
        ("n_tile", ctypes.c_int32), ("tile_bytes", ctypes.c_int32),
        ("w13", ctypes.c_void_p), ("w13_bytes", ctypes.c_size_t),
        ("w2", ctypes.c_void_p), ("w2_bytes", ctypes.c_size_t),
        ("alpha13", ctypes.c_void_p), ("alpha2", ctypes.c_void_p),
        ("scale_mul", ctypes.c_uint32), ("scale_add", ctypes.c_uint32),
        ("layout", ctypes.c_int32),
        ("w13_scales", ctypes.c_void_p), ("w13_scales_bytes", ctypes.c_size_t),
        ("w2_scales", ctypes.c_void_p), ("w2_scales_bytes", ctypes.c_size_t),
    ]


def variant() -> str:
    """Library variant this process loads: "checked" when FP4MOE_BOUNDS_CHECK
    is set to a non-empty value other than 0, else "release"."""
    v = os.environ.get("FP4MOE_BOUNDS_CHECK", "")
    return "checked" if v not in ("", "0") else "release"


def build(force: bool = False, variant_name: str | None = None) -> str:
    """Compile the CUDA library for sm_103a (in-tree): the variant this
    process loads unless one is named."""
    return _build.build(force=force, variant=variant_name or variant())


def exported_symbols() -> list[str]:
    """Function names the C header declares."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"\b(fp4moe_[a-z0-9_]+)\s*\(", text)))


def load() -> ctypes.CDLL:
    """Load libfp4moe.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.lib_path(variant())
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "block_scaled_fp4_02_gb300.build() (needs nvcc)")
        L = ctypes.CDLL(path)
        vp, sz, i32, i64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                            ctypes.c_int64)
        sigs = {
            "fp4moe_requant_fp4_gran_k": (i32, [vp, vp, i64, i64, i32, i32, vp,
                                                vp, vp]),
            "fp4moe_act_quant": (i32, [vp, i64, i64, vp, vp, vp]),
            "fp4moe_prepare_weights": (i32, [vp, vp, vp, vp, vp, vp, i32, i32,
                                             i32, i32, i32, i32, vp,
                                             ctypes.POINTER(vp)]),
            "fp4moe_free_packed": (None, [vp]),
            "fp4moe_packed_info": (i32, [vp, ctypes.POINTER(PackedDesc)]),
            "fp4moe_moe_workspace_size": (sz, [vp, i32, i32]),
            "fp4moe_moe_forward": (i32, [vp, vp, vp, i32, vp, i32, vp, vp, sz,
                                         vp]),
            "fp4moe_moe_workspace_size_host": (sz, [vp, i32, i32]),
            "fp4moe_moe_forward_host": (i32, [vp, vp, vp, i32, vp, i32, vp, vp,
                                              sz, vp]),
            "fp4moe_route_workspace_size": (sz, [i32, i32, i32]),
            "fp4moe_route_debug": (i32, [vp, i32, i32, i32, vp, vp, vp, vp, vp,
                                         vp, vp, sz, vp]),
            "fp4moe_status_string": (ctypes.c_char_p, [i32]),
            "fp4moe_last_device_error": (i32, []),
            "fp4moe_set_stage_events": (i32, [ctypes.POINTER(vp), i32]),
            "fp4moe_moe_workspace_offsets": (i32, [vp, i32, i32,
                                                   ctypes.POINTER(sz), i32]),
            "fp4moe_test_wait_timeout": (i32, [ctypes.c_uint64, vp]),
            "fp4moe_test_bounds_check": (i32, [i64, vp]),
            "fp4moe_build_flags": (i32, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_string(code: int) -> str:
    try:
        return load().fp4moe_status_string(code).decode()
    except Exception:  # library not loadable: still give a message
        return {0: "ok", 1: "invalid argument", 2: "unsupported",
                3: "workspace too small", 4: "CUDA error",
                5: "device wait timed out",
                6: "index out of bounds (bounds-checked build)"}.get(
                    code, "unknown status")


def _check(code: int, what: str) -> None:
    if code != OK:
        raise FP4MoEError(code, what)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _u8(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must be torch.uint8")
    return t


STAGE_EVENTS = 8
STAGE_NAMES = ("route", "scan", "scatter_gather", "fc1_swiglu", "h_fp8_round",
               "fc2", "combine")


def set_stage_events(events) -> None:
    """Hand 8 torch.cuda.Event(enable_timing=True) objects to the next
    moe_forward call on this thread (None clears)."""
    if events is None:
        _check(load().fp4moe_set_stage_events(None, 0), "set_stage_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().fp4moe_set_stage_events(arr, len(events)),
           "set_stage_events")


def last_device_error() -> int:
    """Reads and clears the device status word (synchronises)."""
    return load().fp4moe_last_device_error()


def test_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launches the bounded-wait self-test: a wait on an mbarrier that nothing
    completes gives up after limit_ns and records ERR_TIMEOUT in the device
    status word (read it with last_device_error())."""
    _check(load().fp4moe_test_wait_timeout(limit_ns, _stream(stream)),
           "test_wait_timeout")


def test_bounds_check(index: int, stream=None) -> None:
    """Launches the index-check self-test: slot `index` of a 64-entry device
    array is written through the check of the bounds-checked build; outside
    [0, 64) it records ERR_BOUNDS (read it with last_device_error())."""
    _check(load().fp4moe_test_bounds_check(index, _stream(stream)),
           "test_bounds_check")


def build_flags() -> int:
    """BUILD_BOUNDS_CHECK if the loaded library is the bounds-checked one."""
    return int(load().fp4moe_build_flags())


# ------------------------------------------------------------------- steps

def requant_fp4_gran_k(fp4: torch.Tensor, e4m3_scales: torch.Tensor,
                       fp4_out: torch.Tensor | None = None,
                       ue8m0_out: torch.Tensor | None = None, stream=None):
    """group16 -> group32 requant on the GPU: [rows, K/2] codes + [rows, K/16]
    E4M3 scales -> [rows, K/2] codes + [rows, K/32] UE8M0 scales."""
    _u8(fp4, "fp4")
    if e4m3_scales.dtype == torch.float8_e4m3fn:
        e4m3_scales = e4m3_scales.view(torch.uint8)
    _u8(e4m3_scales, "e4m3_scales")
    rows = fp4.numel() // fp4.shape[-1]
    K = fp4.shape[-1] * 2
    if fp4_out is None:
        fp4_out = torch.empty_like(fp4)
    if ue8m0_out is None:
        ue8m0_out = torch.empty(*fp4.shape[:-1], K // 32, dtype=torch.uint8,
                                device=fp4.device)
    _check(load().fp4moe_requant_fp4_gran_k(
        _ptr(fp4), _ptr(e4m3_scales), rows, K, 16, 32, _ptr(fp4_out),
        _ptr(ue8m0_out), _stream(stream)), "requant_fp4_gran_k")
    return fp4_out, ue8m0_out


def act_quant(x: torch.Tensor, xq: torch.Tensor | None = None,
              xs: torch.Tensor | None = None, stream=None):
    """bf16 [T, K] -> E4M3 [T, K] (uint8) + UE8M0 [T, K/32] (uint8)."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be torch.bfloat16")
    T, K = x.shape
    if xq is None:
        xq = torch.empty(T, K, dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty(T, K // 32, dtype=torch.uint8, device=x.device)
    _check(load().fp4moe_act_quant(_ptr(x), T, K, _ptr(xq), _ptr(xs),
                                   _stream(stream)), "act_quant")
    return xq, xs


def route_workspace_size(T: int, E: int, top_k: int) -> int:
    return load().fp4moe_route_workspace_size(T, E, top_k)


def route_debug(logits: torch.Tensor, top_k: int, stream=None) -> dict:
    """Routing (S2) and permutation (S3) alone, for bit-exact checks."""
    if logits.dtype != torch.float32:
        raise TypeError("logits must be torch.float32")
    T, E = logits.shape
    dev = logits.device
    P = T * top_k
    out = dict(
        ids=torch.empty(T, top_k, dtype=torch.int32, device=dev),
        w=torch.empty(T, top_k, dtype=torch.float32, device=dev),
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm=torch.empty(P, dtype=torch.int32, device=dev),
        inv=torch.empty(P, dtype=torch.int32, device=dev))
    n = route_workspace_size(T, E, top_k)
    if n == 0:
        raise FP4MoEError(ERR_INVALID_ARG, "route_debug")
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    _check(load().fp4moe_route_debug(
        _ptr(logits), T, E, top_k, _ptr(out["ids"]), _ptr(out["w"]),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
        _ptr(out["inv"]), _ptr(ws), n, _stream(stream)), "route_debug")
    return out


class PackedWeights:
    """Prepared weights owned by the library (freed with the object)."""

    def __init__(self, handle: int, keepalive=()):
        self._h = ctypes.c_void_p(handle)
        d = PackedDesc()
        _check(load().fp4moe_packed_info(self._h, ctypes.byref(d)),
               "packed_info")
        self.desc = d
        self.E, self.K, self.I = d.E, d.K, d.I
        self.gran_k, self.act_mode = d.gran_k, d.act_mode

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise RuntimeError("packed weights already freed")
        return self._h

    def free(self) -> None:
        if self._h is not None and _lib is not None:
            _lib.fp4moe_free_packed(self._h)
        self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def buffers(self) -> dict:
        """The packed device buffers as uint8 / float32 torch tensors (copies)."""
        d = self.desc
        out = {}
        items = [("w13", d.w13, d.w13_bytes), ("w2", d.w2, d.w2_bytes),
                 ("alpha13", d.alpha13, 4 * d.E), ("alpha2", d.alpha2, 4 * d.E)]
        if d.layout == 1:
            items += [("w13_scales", d.w13_scales, d.w13_scales_bytes),
                      ("w2_scales", d.w2_scales, d.w2_scales_bytes)]
        for name, ptr, nbytes in items:
            host = torch.empty(nbytes, dtype=torch.uint8)
            _memcpy_d2h(host, ptr, nbytes)
            out[name] = host.view(torch.float32) if name.startswith("alpha") \
                else host
        return out


def _cudart() -> ctypes.CDLL:
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    raise RuntimeError("libcudart not found")


def _memcpy_d2h(host: torch.Tensor, dptr: int, nbytes: int) -> None:
    torch.cuda.synchronize()
    rt = _cudart()
    rt.cudaMemcpy.restype = ctypes.c_int
    rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_size_t, ctypes.c_int]
    if rt.cudaMemcpy(host.data_ptr(), dptr, nbytes, 2) != 0:  # DeviceToHost
        raise FP4MoEError(ERR_CUDA, "cudaMemcpy")


def prepare_weights(w13, w13_s, w13_gs, w2, w2_s, w2_gs, *, gran_k: int = 16,
                    w13_layout: int = W13_GATE_UP, act_mode: int = ACT_BF16,
                    stream=None) -> PackedWeights:
    """Raw grouped FP4 weights -> packed weights (synchronous)."""
    for n, t in (("w13", w13), ("w13_s", w13_s), ("w2", w2), ("w2_s", w2_s)):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn,
                           getattr(torch, "float8_e8m0fnu", torch.uint8)):
            raise TypeError(f"{n} must be a byte tensor")
    w13_s = w13_s.view(torch.uint8)
    w2_s = w2_s.view(torch.uint8)
    E, twoI, kb = w13.shape
    K, I = kb * 2, twoI // 2
    if w13_gs.dtype != torch.float32 or w2_gs.dtype != torch.float32:
        raise TypeError("global scales must be torch.float32")
    h = ctypes.c_void_p()
    _check(load().fp4moe_prepare_weights(
        _ptr(w13), _ptr(w13_s), _ptr(w13_gs), _ptr(w2), _ptr(w2_s),
        _ptr(w2_gs), E, K, I, gran_k, w13_layout, act_mode, _stream(stream),
        ctypes.byref(h)), "prepare_weights")
    return PackedWeights(h.value)


def moe_workspace_size(packed: PackedWeights, T: int, top_k: int) -> int:
    return load().fp4moe_moe_workspace_size(packed.handle, T, top_k)


WS_FIELDS = ("ids", "w", "counts", "offsets", "perm", "inv", "xperm", "h",
             "o", "total", "h_scales", "h_format", "pitch")


def moe_workspace_offsets(packed: PackedWeights, T: int, top_k: int) -> dict:
    """Byte offsets of moe_forward's intermediates inside its workspace
    (plus the h format: 0 bf16, 1 E4M3 bytes + scale words of `pitch`)."""
    n = len(WS_FIELDS)
    arr = (ctypes.c_size_t * n)()
    _check(load().fp4moe_moe_workspace_offsets(packed.handle, T, top_k, arr,
                                               n), "moe_workspace_offsets")
    return dict(zip(WS_FIELDS, list(arr)))


def moe_workspace_size_host(packed: PackedWeights, T: int, top_k: int) -> int:
    return load().fp4moe_moe_workspace_size_host(packed.handle, T, top_k)


def moe_forward(x: torch.Tensor, x_scales: torch.Tensor | None,
                router_logits: torch.Tensor, packed: PackedWeights, top_k: int,
                y: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None):
    """MoE layer forward on device tensors; returns y bf16 [T, K]."""
    T = router_logits.shape[0]
    if router_logits.dtype != torch.float32:
        raise TypeError("router_logits must be torch.float32")
    if y is None:
        y = torch.empty(T, packed.K, dtype=torch.bfloat16, device=x.device)
    n = moe_workspace_size(packed, T, top_k)
    if workspace is None:
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=x.device)
    _check(load().fp4moe_moe_forward(
        _ptr(x), _ptr(x_scales), _ptr(router_logits), T, packed.handle, top_k,
        _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
        "moe_forward")
    return y


def moe_forward_host(x_host: torch.Tensor, x_scales_host: torch.Tensor | None,
                     logits_host: torch.Tensor, packed: PackedWeights,
                     top_k: int, y_host: torch.Tensor, workspace: torch.Tensor,
                     stream=None) -> torch.Tensor:
    """End-to-end call on (pinned) host tensors; asynchronous on the stream."""
    T = logits_host.shape[0]
    for t in (x_host, logits_host, y_host) + (
            (x_scales_host,) if x_scales_host is not None else ()):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    _check(load().fp4moe_moe_forward_host(
        x_host.data_ptr(),
        None if x_scales_host is None else x_scales_host.data_ptr(),
        logits_host.data_ptr(), T, packed.handle, top_k, y_host.data_ptr(),
        _ptr(workspace), workspace.numel(), _stream(stream)),
        "moe_forward_host")
    return y_host
