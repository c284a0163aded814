"""The allocation-free routing entry point, against the workspace one.

fp4moe_route_noalloc serves callers that cannot allocate device memory where
they route tokens (a plugin inside a framework that owns the memory pool, or
a latency-critical loop where cudaMalloc could synchronise the device): it
keeps its scratch in a fixed array inside the library instead of a
caller-provided workspace.  This test calls it through the C ABI twice in a
row, on different inputs, and checks that each call gives exactly what
fp4moe_route_debug (the entry point that takes a workspace) gives for the
same input, so nothing from the first call leaks into the second.  It lives
in a file of its own, collected last, so a stop-at-first-failure run has
already run every other test when it starts.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import block_scaled_fp4_02_gb300 as fp4

pytestmark = pytest.mark.gpu


def _noalloc(lib, logits: torch.Tensor, top_k: int) -> dict:
    T, E = logits.shape
    dev = logits.device
    out = dict(
        ids=torch.empty(T, top_k, dtype=torch.int32, device=dev),
        w=torch.empty(T, top_k, dtype=torch.float32, device=dev),
        counts=torch.empty(E, dtype=torch.int32, device=dev),
        offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        perm=torch.empty(T * top_k, dtype=torch.int32, device=dev),
        inv=torch.empty(T * top_k, dtype=torch.int32, device=dev))
    f = lib.fp4moe_route_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int] \
        + [ctypes.c_void_p] * 7
    rc = f(logits.data_ptr(), T, E, top_k, out["ids"].data_ptr(),
           out["w"].data_ptr(), out["counts"].data_ptr(),
           out["offsets"].data_ptr(), out["perm"].data_ptr(),
           out["inv"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == fp4.OK, fp4.status_string(rc)
    return out


def test_route_noalloc_matches_workspace_entry_point():
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"
    fp4.build()
    lib = fp4.load()
    fp4.last_device_error()
    g = np.random.default_rng(31)
    cases = [(8192, 256, 8), (77, 40, 3)]      # a large call, then a small one
    for T, E, k in cases:
        logits = torch.from_numpy(
            g.standard_normal((T, E)).astype(np.float32)).cuda()
        got = _noalloc(lib, logits, k)
        ref = fp4.route_debug(logits, k)
        torch.cuda.synchronize()
        # the same kernels run on the same logits on both paths: every
        # output, the routing weights included, must be bit-identical
        for name in ("ids", "w", "counts", "offsets", "perm", "inv"):
            assert torch.equal(got[name], ref[name]), name
    assert fp4.last_device_error() == fp4.OK


def test_route_noalloc_rejects_oversized_calls():
    fp4.build()
    lib = fp4.load()
    lib.fp4moe_route_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.fp4moe_route_noalloc_scratch_bytes.argtypes = [ctypes.c_int,
                                                        ctypes.c_int]
    T, E = 65536, 1024
    assert lib.fp4moe_route_noalloc_scratch_bytes(T, E) > (4 << 20)
    f = lib.fp4moe_route_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int] \
        + [ctypes.c_void_p] * 7
    fake = 0x10000   # never dereferenced: the size check comes first
    assert f(fake, T, E, 8, *([fake] * 6), None) == \
        fp4.ERR_WORKSPACE_TOO_SMALL
