"""GPU parity of the integer-exact steps against the oracle: requant (S1),
FP8 activation quantization (S4), routing ids and permutation (S2, S3)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_scaled_fp4_02_gb300 as fp4
import synth
from _util import bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    fp4.build()
    fp4.load()
    assert fp4.build_flags() == (fp4.BUILD_BOUNDS_CHECK
                                 if fp4.variant() == "checked" else 0)
    assert fp4.last_device_error() == fp4.OK


FINITE_E4M3 = np.array([b for b in range(256) if b not in (0x7F, 0xFF)],
                       dtype=np.uint8)


def gpu_requant(codes: np.ndarray, scales: np.ndarray):
    c = torch.from_numpy(codes).cuda()
    s = torch.from_numpy(scales).cuda()
    oc, os_ = fp4.requant_fp4_gran_k(c, s)
    torch.cuda.synchronize()
    return oc.cpu().numpy(), os_.cpu().numpy()


# ------------------------------------------------------------------ requant

def test_requant_every_code_and_scale(orc):
    # Uniform random code bytes and every finite E4M3 scale, K with a ragged
    # number of 32-groups per row.
    rows, K = 4099, 480
    codes = synth.random_bytes((rows, K // 2), 11)
    g = np.random.default_rng(12)
    scales = g.choice(FINITE_E4M3, size=(rows, K // 16))
    scales[:254, 0] = FINITE_E4M3   # each scale at least once
    scales[300:310] = 0            # all-zero scales
    ref_c, ref_s = orc.requant(codes, scales)
    got_c, got_s = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got_s, ref_s)
    np.testing.assert_array_equal(got_c, ref_c)
    assert fp4.last_device_error() == fp4.OK


def test_requant_zero_half_beside_tiny_half(orc):
    # One 16-half all +-0 codes under every finite scale, the other half
    # tiny values under the smallest scales: the group exponent is then far
    # below the zero half's scale (s / 2^e up to 448 * 2^13), which must
    # still give +-0 codes with their signs kept.
    n = FINITE_E4M3.size
    g = np.random.default_rng(21)
    codes = np.empty((n, 16), dtype=np.uint8)
    codes[:, :8] = g.choice(np.array([0x00, 0x08, 0x80, 0x88], dtype=np.uint8),
                            size=(n, 8))
    codes[:, 8:] = g.integers(0, 256, size=(n, 8), dtype=np.uint8) & 0x99
    scales = np.empty((n, 2), dtype=np.uint8)
    scales[:, 0] = FINITE_E4M3
    scales[:, 1] = g.choice(np.array([0x01, 0x02, 0x81, 0x09], dtype=np.uint8), size=n)
    # the same with the halves swapped
    codes = np.concatenate([codes, np.concatenate([codes[:, 8:], codes[:, :8]], 1)])
    scales = np.concatenate([scales, scales[:, ::-1]])
    ref_c, ref_s = orc.requant(codes, scales)
    got_c, got_s = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got_s, ref_s)
    np.testing.assert_array_equal(got_c, ref_c)
    assert fp4.last_device_error() == fp4.OK


def test_requant_nan_scale(orc):
    codes = synth.random_bytes((8, 64), 13)
    scales = np.full((8, 8), 0x38, dtype=np.uint8)
    scales[3, 5] = 0x7F
    scales[6, 0] = 0xFF
    ref_c, ref_s = orc.requant(codes, scales)
    got_c, got_s = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got_s, ref_s)
    np.testing.assert_array_equal(got_c, ref_c)
    assert got_s[3, 2] == 0xFF and got_s[6, 0] == 0xFF
    assert fp4.last_device_error() == fp4.ERR_INVALID_ARG
    assert fp4.last_device_error() == fp4.OK   # read-and-clear


@pytest.mark.parametrize("rows,K", [(1, 32), (7, 64), (33, 96)])
def test_requant_tiny_shapes(orc, rows, K):
    codes = synth.random_bytes((rows, K // 2), rows * K)
    scales = np.random.default_rng(rows).choice(FINITE_E4M3, size=(rows, K // 16))
    ref = orc.requant(codes, scales)
    got = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


def test_requant_small_config(orc):
    codes, scales, _ = synth.requant_inputs(synth.SMALL_REQUANT)
    ref = orc.requant(codes, scales)
    got = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


def test_requant_full_size_bit_exact(orc):
    # [32 x 4096, 7168] with 0.1% x20 outliers, every output byte compared.
    codes, scales, _ = synth.requant_inputs(synth.REQUANT)
    ref_c, ref_s = orc.requant(codes, scales)
    got_c, got_s = gpu_requant(codes, scales)
    np.testing.assert_array_equal(got_s, ref_s)
    assert np.array_equal(got_c, ref_c), int((got_c != ref_c).sum())
    assert fp4.last_device_error() == fp4.OK


# ------------------------------------------------------------ act quant

@pytest.mark.parametrize("T,K", [(1, 32), (37, 512), (4096, 7168)])
def test_act_quant_bit_exact(orc, T, K):
    g = np.random.default_rng(T + K)
    x = g.standard_normal((T, K)).astype(np.float32)
    x[0, :32] = 0.0
    if T > 4:
        x[1] *= 1e-30
        x[2] *= 1e30
        x[3, :64] = -0.0
    xb = synth.f32_to_bf16_bits(x)
    ref_q, ref_s = orc.act_quant(xb)
    q, s = fp4.act_quant(bf16_tensor(xb))
    np.testing.assert_array_equal(s.cpu().numpy(), ref_s)
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)
    assert fp4.last_device_error() == fp4.OK


def test_act_quant_fp8_workload(orc):
    a = synth.moe_activations(synth.FP8)
    ref_q, ref_s = orc.act_quant(a["x_bf16"])
    q, s = fp4.act_quant(bf16_tensor(a["x_bf16"]))
    np.testing.assert_array_equal(s.cpu().numpy(), ref_s)
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)


# ---------------------------------------------------------------- routing

def check_route(orc, logits: np.ndarray, k: int):
    E = logits.shape[1]
    got = fp4.route_debug(torch.from_numpy(logits).cuda(), k)
    torch.cuda.synchronize()
    ids, w = orc.route(logits, k)
    counts, offsets, perm, inv = orc.permute(ids, E)
    np.testing.assert_array_equal(got["ids"].cpu().numpy(), ids)
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(got["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(got["perm"].cpu().numpy(), perm)
    np.testing.assert_array_equal(got["inv"].cpu().numpy(), inv)
    np.testing.assert_allclose(got["w"].cpu().numpy(), w, rtol=1e-6, atol=1e-7)
    assert fp4.last_device_error() == fp4.OK


@pytest.mark.parametrize("cfg", [synth.TINY, synth.SMALL_DECODE,
                                 synth.SMALL_PREFILL, synth.SMALL_FP8,
                                 synth.DECODE, synth.DECODE_SKEW,
                                 synth.PREFILL, synth.FP8],
                         ids=lambda c: c.name)
def test_route_workloads(orc, cfg):
    check_route(orc, synth.moe_activations(cfg)["logits"], cfg.top_k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 8, 8), (33, 40, 3),
                                   (70, 1024, 16), (1000, 96, 7)])
def test_route_shapes(orc, T, E, k):
    logits = np.random.default_rng(T * E + k).standard_normal((T, E)).astype(
        np.float32)
    check_route(orc, logits, k)


def test_route_ties(orc):
    # Many exactly equal logits: the lower expert id must win every tie.
    g = np.random.default_rng(21)
    logits = g.integers(0, 3, size=(500, 64)).astype(np.float32)
    logits[7] = 1.0
    check_route(orc, logits, 6)


def test_route_nan_logit_is_reported():
    logits = torch.zeros(4, 16, device="cuda")
    logits[2, 3] = float("nan")
    fp4.route_debug(logits, 2)
    assert fp4.last_device_error() == fp4.ERR_INVALID_ARG


# ------------------------------------------------------- bounded device waits

def test_bounded_wait_gives_up_and_records_timeout():
    # A wait on an mbarrier that nothing completes gives up after its limit
    # (1 ms here; the library's kernels use about 2 s) and records TIMEOUT in
    # the status word; the context stays usable afterwards.
    assert fp4.last_device_error() == fp4.OK
    fp4.test_wait_timeout(1_000_000)
    torch.cuda.synchronize()
    assert fp4.last_device_error() == fp4.ERR_TIMEOUT
    assert fp4.last_device_error() == fp4.OK      # read clears it
    x = torch.arange(64, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 2016.0
    codes, scales, _ = synth.requant_inputs(synth.SMALL_REQUANT)
    gpu_requant(codes, scales)
    assert fp4.last_device_error() == fp4.OK


# ------------------------------------------------------------- index checks

@pytest.mark.parametrize("index,expect", [(0, fp4.OK), (63, fp4.OK),
                                          (64, fp4.ERR_BOUNDS),
                                          (-1, fp4.ERR_BOUNDS),
                                          (1 << 40, fp4.ERR_BOUNDS)])
def test_index_check_records_bounds_and_skips_the_access(index, expect):
    # The check the bounds-checked build applies to every data-dependent
    # index, run on a 64-entry array: out of range it records BOUNDS and
    # writes nothing (the context stays usable).
    assert fp4.last_device_error() == fp4.OK
    fp4.test_bounds_check(index)
    torch.cuda.synchronize()
    assert fp4.last_device_error() == expect
    x = torch.arange(64, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 2016.0
