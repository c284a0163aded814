"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before launching anything."""
from __future__ import annotations

import ctypes

import pytest

import block_scaled_fp4_02_gb300 as fp4


@pytest.fixture(scope="module")
def lib():
    fp4.build()
    return fp4.load()


def test_exports_every_header_symbol(lib):
    names = fp4.exported_symbols()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported"),
                       (3, "workspace too small"), (4, "CUDA error"),
                       (5, "device wait timed out"),
                       (6, "index out of bounds (bounds-checked build)"),
                       (99, "unknown status")]:
        assert lib.fp4moe_status_string(code).decode() == text


def test_bounds_checked_variant_builds_and_exports_every_symbol():
    # The same sources compiled with FP4MOE_BOUNDS_CHECK; both variants say
    # which they are (a host-only call).
    import importlib
    b = importlib.import_module("block_scaled_fp4_02_gb300.build")
    path = fp4.build(variant_name="checked")
    assert path == b.lib_path("checked") and path != b.lib_path("release")
    checked = ctypes.CDLL(path)
    missing = [n for n in fp4.exported_symbols() if not hasattr(checked, n)]
    assert not missing, missing
    assert checked.fp4moe_build_flags() == fp4.BUILD_BOUNDS_CHECK
    assert ctypes.CDLL(b.lib_path("release")).fp4moe_build_flags() == 0


def test_variant_follows_the_environment(monkeypatch):
    monkeypatch.delenv("FP4MOE_BOUNDS_CHECK", raising=False)
    assert fp4.variant() == "release"
    monkeypatch.setenv("FP4MOE_BOUNDS_CHECK", "0")
    assert fp4.variant() == "release"
    monkeypatch.setenv("FP4MOE_BOUNDS_CHECK", "1")
    assert fp4.variant() == "checked"


FAKE = 0x10000  # an aligned non-null address; never dereferenced on the host


def test_requant_argument_checks(lib):
    f = lib.fp4moe_requant_fp4_gran_k
    assert f(FAKE, FAKE, 4, 48, 16, 32, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 64, 32, 16, FAKE, FAKE, None) == fp4.ERR_UNSUPPORTED
    assert f(FAKE, FAKE, 4, 64, 16, 8, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(FAKE, FAKE, -1, 64, 16, 32, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(None, FAKE, 4, 64, 16, 32, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(FAKE + 8, FAKE, 4, 64, 16, 32, FAKE, FAKE, None) == \
        fp4.ERR_INVALID_ARG                      # misaligned codes
    assert f(FAKE, FAKE, 0, 64, 16, 32, FAKE, FAKE, None) == fp4.OK  # no-op


def test_act_quant_argument_checks(lib):
    f = lib.fp4moe_act_quant
    assert f(FAKE, 4, 48, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(None, 4, 64, FAKE, FAKE, None) == fp4.ERR_INVALID_ARG
    assert f(FAKE, 0, 64, FAKE, FAKE, None) == fp4.OK


def test_route_argument_checks(lib):
    assert lib.fp4moe_route_workspace_size(8, 0, 1) == 0
    assert lib.fp4moe_route_workspace_size(8, 4, 5) == 0
    assert lib.fp4moe_route_workspace_size(8, 64, 17) == 0
    assert lib.fp4moe_route_workspace_size(8, 2048, 2) == 0
    n = lib.fp4moe_route_workspace_size(100, 64, 8)
    assert n > 0 and n % 256 == 0
    f = lib.fp4moe_route_debug
    args = [FAKE] * 6
    assert f(FAKE, 10, 8, 9, *args, FAKE, 1 << 20, None) == fp4.ERR_INVALID_ARG
    assert f(FAKE, 10, 8, 2, *args, FAKE, 16, None) == \
        fp4.ERR_WORKSPACE_TOO_SMALL
    assert f(FAKE, 10, 8, 2, *args, FAKE + 16, 1 << 20, None) == \
        fp4.ERR_INVALID_ARG                      # workspace alignment


def _prepare(lib, **kw):
    a = dict(w13=FAKE, w13_s=FAKE, w13_gs=FAKE, w2=FAKE, w2_s=FAKE,
             w2_gs=FAKE, E=4, K=256, I=128, gran=16, layout=0, act=0)
    a.update(kw)
    out = ctypes.c_void_p(123)
    rc = lib.fp4moe_prepare_weights(
        a["w13"], a["w13_s"], a["w13_gs"], a["w2"], a["w2_s"], a["w2_gs"],
        a["E"], a["K"], a["I"], a["gran"], a["layout"], a["act"], None,
        ctypes.byref(out))
    return rc, out


def test_prepare_argument_checks(lib):
    for kw in [dict(gran=8), dict(layout=2), dict(act=3), dict(K=192),
               dict(I=64), dict(E=0), dict(w2=None), dict(act=0x800)]:
        rc, out = _prepare(lib, **kw)
        assert rc == fp4.ERR_INVALID_ARG, kw
        assert not out.value
    # FP8 activations over group16 scales without the lossy requant: refused,
    # like the fused-compute capability gate for recipe (1,1,16).
    rc, out = _prepare(lib, act=fp4.ACT_FP8 | fp4.FLAG_NO_REQUANT, gran=16)
    assert rc == fp4.ERR_UNSUPPORTED and not out.value
    # The exact-group16 flag is a known bit: a bad shape is still reported
    # as such (these checks never reach the device).
    rc, out = _prepare(lib, act=fp4.ACT_FP8 | fp4.FLAG_KEEP_GROUP16, gran=16, K=192)
    assert rc == fp4.ERR_INVALID_ARG and not out.value


def test_moe_argument_checks(lib):
    assert lib.fp4moe_moe_workspace_size(None, 8, 2) == 0
    assert lib.fp4moe_moe_forward(FAKE, None, FAKE, 8, None, 2, FAKE, FAKE,
                                  1 << 20, None) == fp4.ERR_INVALID_ARG
    assert lib.fp4moe_moe_forward_host(FAKE, None, FAKE, 8, None, 2, FAKE,
                                       FAKE, 1 << 20, None) == \
        fp4.ERR_INVALID_ARG


def test_wait_timeout_argument_checks(lib):
    f = lib.fp4moe_test_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    assert f(0, None) == fp4.ERR_INVALID_ARG
    assert f(2_000_000_000, None) == fp4.ERR_INVALID_ARG
