"""FP64 CPU oracle for the block-scaled FP4 MoE hot path (test infrastructure).

Only tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The product (``block_scaled_fp4_02_gb300``) never imports it, and
the two share no code.  The arithmetic lives in ``oracle.cpp``; this module
compiles it with the host compiler and wraps it with ctypes.

Each function cites, in ``oracle.cpp``, the passage of the pages it follows.
Every function is pinned by tests/test_oracle_pins.py (closed forms,
invariants, brute force on tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into a shared library (portable flags, no -march)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class _OrcMoe(ctypes.Structure):
    _fields_ = [
        ("w13", ctypes.c_void_p), ("w13_s", ctypes.c_void_p),
        ("w13_gs", ctypes.c_void_p), ("w2", ctypes.c_void_p),
        ("w2_s", ctypes.c_void_p), ("w2_gs", ctypes.c_void_p),
        ("E", ctypes.c_int32), ("K", ctypes.c_int32), ("I", ctypes.c_int32),
        ("gran", ctypes.c_int32), ("w13_layout", ctypes.c_int32),
        ("act_mode", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("nthreads", ctypes.c_int32),
        ("x_bf16", ctypes.c_void_p), ("xq", ctypes.c_void_p),
        ("xs", ctypes.c_void_p), ("logits", ctypes.c_void_p),
        ("T", ctypes.c_int64), ("h_out", ctypes.c_void_p),
        ("aux_out", ctypes.c_void_p),
    ]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            L = _lib
            L.orc_e2m1_value.restype = ctypes.c_double
            L.orc_e2m1_value.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_value.restype = ctypes.c_double
            L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            L.orc_ue8m0_value.restype = ctypes.c_double
            L.orc_ue8m0_value.argtypes = [ctypes.c_uint8]
            L.orc_bf16_value.restype = ctypes.c_double
            L.orc_bf16_value.argtypes = [ctypes.c_uint16]
            L.orc_e2m1_rne.restype = ctypes.c_uint8
            L.orc_e2m1_rne.argtypes = [ctypes.c_double]
            L.orc_e4m3_rne_sat.restype = ctypes.c_uint8
            L.orc_e4m3_rne_sat.argtypes = [ctypes.c_double]
            L.orc_bf16_rne.restype = ctypes.c_uint16
            L.orc_bf16_rne.argtypes = [ctypes.c_double]
            L.orc_requant.restype = ctypes.c_int
            L.orc_requant.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int]
            L.orc_route.restype = ctypes.c_int
            L.orc_route.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p]
            L.orc_permute.restype = ctypes.c_int
            L.orc_permute.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_int, ctypes.c_int] + \
                [ctypes.c_void_p] * 4
            L.orc_act_quant.restype = ctypes.c_int
            L.orc_act_quant.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_void_p]
            L.orc_round_intermediate.restype = ctypes.c_int
            L.orc_round_intermediate.argtypes = [ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_int,
                                                 ctypes.c_void_p]
            L.orc_fp8_group_exponent.restype = ctypes.c_int
            L.orc_fp8_group_exponent.argtypes = [ctypes.c_void_p]
            L.orc_moe_rows.restype = ctypes.c_int
            L.orc_moe_rows.argtypes = [ctypes.POINTER(_OrcMoe),
                                       ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_void_p]
        return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ------------------------------------------------------------------ scalars

def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e4m3_value(b: int) -> float:
    return lib().orc_e4m3_value(b)


def ue8m0_value(b: int) -> float:
    return lib().orc_ue8m0_value(b)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def e2m1_rne(v: float) -> int:
    return lib().orc_e2m1_rne(v)


def e4m3_rne_sat(v: float) -> int:
    return lib().orc_e4m3_rne_sat(v)


def bf16_rne(v: float) -> int:
    return lib().orc_bf16_rne(v)


def bf16_rne_array(v: np.ndarray) -> np.ndarray:
    """bfloat16 bits (uint16) of an FP64 array, one oracle call per element."""
    f = lib().orc_bf16_rne
    flat = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.fromiter((f(float(x)) for x in flat), dtype=np.uint16,
                      count=flat.size)
    return out.reshape(np.shape(v))


# ------------------------------------------------------------------- steps

def requant(fp4: np.ndarray, s16: np.ndarray, nthreads: int | None = None):
    """group16 -> group32 requant (S1).  fp4 [rows, K/2] u8, s16 [rows, K/16]."""
    fp4 = np.ascontiguousarray(fp4, dtype=np.uint8)
    s16 = np.ascontiguousarray(s16, dtype=np.uint8)
    rows, kb = fp4.shape
    K = kb * 2
    assert s16.shape == (rows, K // 16)
    out = np.empty_like(fp4)
    s32 = np.empty((rows, K // 32), dtype=np.uint8)
    rc = lib().orc_requant(_ptr(fp4), _ptr(s16), rows, K, _ptr(out),
                           _ptr(s32), nthreads or cores())
    if rc:
        raise ValueError("oracle requant rejected its input")
    return out, s32


def route(logits: np.ndarray, top_k: int):
    """Softmax top-k routing (S2).  Returns ids [T,k] int32, w [T,k] float64."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    if lib().orc_route(_ptr(logits), T, E, top_k, _ptr(ids), _ptr(w)):
        raise ValueError("oracle route rejected its input")
    return ids, w


def permute(ids: np.ndarray, E: int):
    """Stable expert-major permutation (S3): counts, offsets, perm, inv."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    if lib().orc_permute(_ptr(ids), T, k, E, _ptr(counts), _ptr(offsets),
                         _ptr(perm), _ptr(inv)):
        raise ValueError("oracle permute rejected its input")
    return counts, offsets, perm, inv


def act_quant(x_bf16: np.ndarray):
    """FP8 E4M3 + UE8M0/32 activation quantization (S4).  x: uint16 bf16 bits."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, K = x_bf16.shape
    q = np.empty((T, K), dtype=np.uint8)
    s = np.empty((T, K // 32), dtype=np.uint8)
    if lib().orc_act_quant(_ptr(x_bf16), T, K, _ptr(q), _ptr(s)):
        raise ValueError("oracle act_quant rejected its input")
    return q, s


def round_intermediate(h: np.ndarray, act_mode: int) -> np.ndarray:
    """h rounded as stored between FC1 and FC2 (bf16, or E4M3 x UE8M0/32)."""
    h = np.ascontiguousarray(h, dtype=np.float64)
    out = np.empty_like(h)
    if lib().orc_round_intermediate(_ptr(h), h.size, act_mode, _ptr(out)):
        raise ValueError("oracle round_intermediate rejected its input")
    return out


def fp8_group_exponent(h32: np.ndarray) -> int:
    h32 = np.ascontiguousarray(h32, dtype=np.float64)
    assert h32.size == 32
    return lib().orc_fp8_group_exponent(_ptr(h32))


def moe_rows(tokens, *, w13, w13_s, w13_gs, w2, w2_s, w2_gs, gran,
             w13_layout, act_mode, top_k, logits, x_bf16=None, xq=None,
             xs=None, nthreads=None, return_h=False):
    """MoE output rows y[t] in FP64 (before the final bf16 rounding), S2-S7.

    With return_h, also returns the unrounded intermediate h [ntok, k, I]
    and aux [ntok, k, I, 6] = (G, U, sum|G terms|, sum|U terms|,
    sum|G running sums|, sum|U running sums|), the running sums taken after
    each chunk of 16 consecutive K terms (FP32 error-analysis quantities)."""
    E, twoI, kb = w13.shape
    K, I = kb * 2, twoI // 2
    T = logits.shape[0]
    arrs = dict(w13=np.ascontiguousarray(w13, dtype=np.uint8),
                w13_s=np.ascontiguousarray(w13_s, dtype=np.uint8),
                w13_gs=np.ascontiguousarray(w13_gs, dtype=np.float32),
                w2=np.ascontiguousarray(w2, dtype=np.uint8),
                w2_s=np.ascontiguousarray(w2_s, dtype=np.uint8),
                w2_gs=np.ascontiguousarray(w2_gs, dtype=np.float32),
                logits=np.ascontiguousarray(logits, dtype=np.float32))
    if act_mode == 0:
        arrs["x_bf16"] = np.ascontiguousarray(x_bf16, dtype=np.uint16)
        arrs["xq"] = arrs["xs"] = None
    else:
        arrs["x_bf16"] = None
        arrs["xq"] = np.ascontiguousarray(xq, dtype=np.uint8)
        arrs["xs"] = np.ascontiguousarray(xs, dtype=np.uint8)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    h = np.empty((tok.size, top_k, I), dtype=np.float64) if return_h else None
    aux = (np.empty((tok.size, top_k, I, 6), dtype=np.float64) if return_h
           else None)
    args = _OrcMoe(
        _ptr(arrs["w13"]), _ptr(arrs["w13_s"]), _ptr(arrs["w13_gs"]),
        _ptr(arrs["w2"]), _ptr(arrs["w2_s"]), _ptr(arrs["w2_gs"]),
        E, K, I, gran, w13_layout, act_mode, top_k, nthreads or cores(),
        _ptr(arrs["x_bf16"]), _ptr(arrs["xq"]), _ptr(arrs["xs"]),
        _ptr(arrs["logits"]), T, _ptr(h), _ptr(aux))
    y = np.empty((tok.size, K), dtype=np.float64)
    if lib().orc_moe_rows(ctypes.byref(args), _ptr(tok), tok.size, _ptr(y)):
        raise ValueError("oracle moe_rows rejected its input")
    return (y, h, aux) if return_h else y
