"""Seeded synthetic inputs for the block-scaled FP4 MoE workloads.

This module draws random numbers and lays them out as the hot path's inputs;
it is shared by the tests, the oracle checks and the benchmark, and it holds
none of the hot path's own arithmetic (no requant, routing, permutation,
GEMM, SwiGLU or combine).

Weights are drawn FP32 N(0, 0.02) and then encoded as NVFP4 (E2M1 codes, one
E4M3 scale per 16 K-elements, one FP32 global scale per expert matrix), which
is the input format the pages' checkpoints arrive in.  That encoding (in
synth.c) is an input recipe, not a step of the method: it rounds to nearest
with ties away from zero through table look-ups, and neither the oracle nor
the CUDA library calls it.  The recipe:

    gs   = amax(W_e) / (6 * 448)                    per expert matrix
    s16  = nearest E4M3 to amax(group16) / (6 * gs)
    code = nearest E2M1 to w / (s16 * gs)            (s16 == 0 -> code 0)

Streams: weights use a counter-based generator keyed by (seed, expert), so
experts generate in parallel and reproducibly; logits and activations use
``numpy.random.SeedSequence(seed).spawn`` children.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

# ---------------------------------------------------------------- workloads


@dataclass(frozen=True)
class MoeConfig:
    name: str
    E: int
    K: int
    I: int
    T: int
    top_k: int
    act: str = "bf16"        # "bf16" (W4A16) or "fp8" (E4M3 + UE8M0/32)
    skew: float = 0.0        # added to the logits of experts 0..15
    weight_seed: int = 0
    input_seed: int = 0
    w13_layout: int = 0      # 0 = gate_up ("w31"), 1 = up_gate ("w13")
    keep_group16: bool = False   # FP8 over the group16 weights as they are

    @property
    def pairs(self) -> int:
        return self.T * self.top_k

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: FC1 (2 x K x 2I) + FC2 (2 x I x K) per pair."""
        return 6 * self.K * self.I * self.pairs


@dataclass(frozen=True)
class RequantConfig:
    name: str
    rows: int
    K: int
    experts: int
    seed: int
    outlier_p: float = 0.001
    outlier_mul: float = 20.0

    @property
    def elements(self) -> int:
        return self.rows * self.K

    @property
    def bytes_moved(self) -> int:
        """0.5 + 1/16 bytes read and 0.5 + 1/32 bytes written per element."""
        n = self.elements
        return n // 2 + n // 16 + n // 2 + n // 32


# The five workloads of the benchmark description, plus small variants that
# the oracle finishes in seconds and that still span several tiles and a
# ragged tail.
TINY = MoeConfig("tiny_w4a16_E8_K256_I128_T16_k2", 8, 256, 128, 16, 2,
                 weight_seed=1001, input_seed=2001)
REQUANT = RequantConfig("requant_g16_to_g32_E32_N4096_K7168", 32 * 4096, 7168,
                        32, 1002)
DECODE = MoeConfig("decode_w4a16_E256_K6144_I2048_T64_k8", 256, 6144, 2048, 64,
                   8, weight_seed=1003, input_seed=2003)
DECODE_SKEW = MoeConfig("decode_skewed_w4a16_E256_K6144_I2048_T64_k8", 256,
                        6144, 2048, 64, 8, skew=2.0, weight_seed=1003,
                        input_seed=2013)
PREFILL = MoeConfig("prefill_w4a16_E256_K6144_I2048_T8192_k8", 256, 6144, 2048,
                    8192, 8, weight_seed=1003, input_seed=2004)
FP8 = MoeConfig("fp8xfp4_E128_K7168_I2048_T4096_k8", 128, 7168, 2048, 4096, 8,
                act="fp8", weight_seed=1005, input_seed=2005)

SMALL_DECODE = MoeConfig("small_decode_E32_K512_I256_T13_k4", 32, 512, 256, 13,
                         4, weight_seed=3001, input_seed=3101)
SMALL_PREFILL = MoeConfig("small_prefill_E8_K768_I384_T700_k2", 8, 768, 384,
                          700, 2, weight_seed=3002, input_seed=3102)
SMALL_FP8 = MoeConfig("small_fp8_E16_K512_I256_T77_k4", 16, 512, 256, 77, 4,
                      act="fp8", weight_seed=3003, input_seed=3103)
SMALL_REQUANT = RequantConfig("small_requant_E3_N100_K480", 3 * 100, 480, 3,
                              3004)

CONFIGS = {c.name: c for c in (TINY, DECODE, DECODE_SKEW, PREFILL, FP8,
                               SMALL_DECODE, SMALL_PREFILL, SMALL_FP8)}

# --------------------------------------------------------------- weights
# The weight generator is portable C (synth.c): SplitMix64 counters, Box-Muller
# normals and the NVFP4 encoding recipe, threaded over experts.

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                    "-ffp-contract=off", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _clib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.synth_nvfp4_weights.restype = ctypes.c_int
        L.synth_nvfp4_weights.argtypes = [
            ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_float, ctypes.c_double, ctypes.c_float, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _lib = L
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _rng(seq: np.random.SeedSequence) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seq))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> bfloat16 bits, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def nvfp4_weights(E: int, N: int, Kd: int, seed: int, outlier_p=0.0,
                  outlier_mul=1.0, threads: int | None = None):
    """E expert matrices [N, Kd] drawn N(0, 0.02) and encoded as NVFP4 g16:
    codes [E, N, Kd/2] u8, E4M3 scales [E, N, Kd/16] u8, gs [E] f32."""
    codes = np.empty((E, N, Kd // 2), dtype=np.uint8)
    scales = np.empty((E, N, Kd // 16), dtype=np.uint8)
    gs = np.empty(E, dtype=np.float32)
    rc = _clib().synth_nvfp4_weights(
        seed & 0xFFFFFFFFFFFFFFFF, E, N, Kd, 0.02, outlier_p, outlier_mul,
        codes.ctypes.data, scales.ctypes.data, gs.ctypes.data,
        threads or _threads())
    if rc:
        raise ValueError("bad weight shape")
    return codes, scales, gs


def moe_weights(cfg: MoeConfig, threads: int | None = None):
    """w13 [E, 2I, K] (gate_up or up_gate rows) and w2 [E, K, I], NVFP4 g16."""
    base = np.random.SeedSequence(cfg.weight_seed).spawn(2)
    s13 = int(base[0].generate_state(1)[0])
    s2 = int(base[1].generate_state(1)[0])
    w13, w13_s, w13_gs = nvfp4_weights(cfg.E, 2 * cfg.I, cfg.K, s13,
                                       threads=threads)
    w2, w2_s, w2_gs = nvfp4_weights(cfg.E, cfg.K, cfg.I, s2, threads=threads)
    return dict(w13=w13, w13_s=w13_s, w13_gs=w13_gs, w2=w2, w2_s=w2_s,
                w2_gs=w2_gs)


def moe_activations(cfg: MoeConfig):
    """Router logits fp32 N(0,1) [T, E] (+skew on experts 0..15) and x bf16
    N(0,1) [T, K] as uint16 bits."""
    s_log, s_x = np.random.SeedSequence(cfg.input_seed).spawn(2)
    logits = _rng(s_log).standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if cfg.skew:
        logits[:, :16] += np.float32(cfg.skew)
    x = _rng(s_x).standard_normal((cfg.T, cfg.K), dtype=np.float32)
    return dict(logits=logits, x_bf16=f32_to_bf16_bits(x))


def requant_inputs(cfg: RequantConfig, threads: int | None = None):
    """[rows, K] weights from N(0,0.02) with outliers, NVFP4 g16 per expert."""
    n = cfg.rows // cfg.experts
    codes, scales, gs = nvfp4_weights(cfg.experts, n, cfg.K, cfg.seed,
                                      outlier_p=cfg.outlier_p,
                                      outlier_mul=cfg.outlier_mul,
                                      threads=threads)
    return (codes.reshape(cfg.rows, cfg.K // 2),
            scales.reshape(cfg.rows, cfg.K // 16), gs)


def random_bytes(shape, seed: int) -> np.ndarray:
    """Uniform random bytes: every code and scale byte, for exhaustive-style
    checks of integer encodings."""
    return _rng(np.random.SeedSequence(seed)).integers(0, 256, size=shape,
                                                       dtype=np.uint8)
