"""Shared helpers for the parity tests (no method arithmetic of their own,
apart from the tolerance rule and the test-side decoder of the packed layout,
which restates the layout specification independently of the packer)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth

# |gpu - oracle| <= 2^-7 * |oracle| + 1e-3 * rms(oracle), per element.
REL_TOL = 2.0 ** -7
RMS_TOL = 1e-3


def tolerance_violations(gpu, ref, rms=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(gpu - ref)
    return err > bound, err, bound, rms


def assert_within_tolerance(gpu, ref, what="", rms=None):
    bad, err, bound, rms = tolerance_violations(gpu, ref, rms)
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside "
            f"|d| <= 2^-7|ref| + 1e-3 rms (rms {rms:.4g}); worst at {i}: "
            f"gpu {np.asarray(gpu)[i]!r} ref {np.asarray(ref)[i]!r}")


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(
        device).view(torch.bfloat16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


@functools.lru_cache(maxsize=2)
def cached_weights(cfg_key):
    """Weights of a MoE config (shared by configs with the same seed/shape)."""
    E, K, I, seed = cfg_key
    cfg = synth.MoeConfig("w", E, K, I, 1, 1, weight_seed=seed)
    return synth.moe_weights(cfg)


def weights_for(cfg):
    return cached_weights((cfg.E, cfg.K, cfg.I, cfg.weight_seed))


def requant_weights_oracle(orc, w, E, K, I):
    """group32 weights by the ORACLE's requant (what the FP8 path consumes)."""
    c13, s13 = orc.requant(w["w13"].reshape(-1, K // 2),
                           w["w13_s"].reshape(-1, K // 16))
    c2, s2 = orc.requant(w["w2"].reshape(-1, I // 2),
                         w["w2_s"].reshape(-1, I // 16))
    return dict(w13=c13.reshape(E, 2 * I, K // 2),
                w13_s=s13.reshape(E, 2 * I, K // 32), w13_gs=w["w13_gs"],
                w2=c2.reshape(E, K, I // 2), w2_s=s2.reshape(E, K, I // 32),
                w2_gs=w["w2_gs"])


# ---------------------------------------------------------------- layout
# Test-side decoder of the packed tile layout (independent of the packer):
# tile (e, nb, ks) = 128 rows x 64 K; bytes [0,4096) data as
# [half][row][16 B], each 16 B = 4 words of 8 elements; bit b of element j's
# E2M1 code (b = 0, 1, 2: magnitude m, e0, e1; b = 3: sign) sits at word bit
# BIT_POS[j][b]; bytes [4096, ...) scale codes [row][64/gran].
BIT_POS = [[14, 7, 8, 15], [30, 23, 24, 31], [0, 1, 2, 9], [16, 17, 18, 25],
           [26, 27, 28, 3], [10, 11, 12, 19], [4, 5, 6, 13], [20, 21, 22, 29]]
E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4,
                 -6])


def decode_packed(buf: np.ndarray, E, N, Kd, gran, smul, sadd, alpha,
                  gated, I=None, layout=0):
    """Packed bytes -> dequantized weights [E, N, Kd] in source row order."""
    nb, ks = N // 128, Kd // 64
    tb = 4096 + 128 * (64 // gran)
    t = buf[: E * nb * ks * tb].reshape(E, nb, ks, tb)
    data = t[..., :4096].reshape(E, nb, ks, 2, 128, 4, 4).copy()
    words = data.view(np.uint32).reshape(E, nb, ks, 2, 128, 4)
    codes = np.zeros((E, nb, ks, 2, 128, 4, 8), dtype=np.uint8)
    for j in range(8):
        c = np.zeros(words.shape, dtype=np.uint32)
        for b in range(4):
            c |= ((words >> np.uint32(BIT_POS[j][b])) & np.uint32(1)) << np.uint32(b)
        codes[..., j] = c.astype(np.uint8)
    # -> [E, nb, 128 rows, ks, 64 k]
    codes = codes.transpose(0, 1, 4, 2, 3, 5, 6).reshape(E, nb, 128, ks, 64)
    sc = t[..., 4096:].reshape(E, nb, ks, 128, 64 // gran).astype(np.uint32)
    sbits = sc * np.uint32(smul) + np.uint32(sadd)          # bf16 bits
    sval = (sbits << np.uint32(16)).view(np.float32).astype(np.float64)
    sval = sval.transpose(0, 1, 3, 2, 4)                   # [E, nb, 128, ks, g]
    sval = np.repeat(sval, gran, axis=-1)                  # per k
    # dequant = e2m1 * 2^-126 * S * alpha
    val = E2M1[codes] * sval * 2.0 ** -126 * alpha[:, None, None, None, None]
    val = val.reshape(E, nb, 128, Kd)
    out = np.empty((E, N, Kd))
    r = np.arange(128)
    for b in range(nb):
        if gated:
            q, l = r // 32, r % 32
            i = 64 * b + 16 * q + (l % 16)
            gate0, up0 = (0, I) if layout == 0 else (I, 0)
            src = np.where(l < 16, gate0 + i, up0 + i)
        else:
            src = 128 * b + r
        out[:, src, :] = val[:, b]
    return out


def decode_packed_mx(codes, words, E, N, Kd, alpha, gated, I=None, layout=0):
    """Block-scaled layout -> dequantized weights [E, N, Kd] in source row
    order.  codes: [E][N][Kd/2] bytes with FC1 rows reordered (per 128-column
    block b: gate rows at 256 b, up rows at 256 b + 128); words: one 32-bit
    word per row and 128-wide step, [E][N/128][Kd/128][128], byte j = UE8M0
    of the step's j-th 32-wide block."""
    c = codes[: E * N * Kd // 2].reshape(E, N, Kd // 2)
    lo, hi = c & 0xF, c >> 4
    e2m1 = E2M1[np.stack([lo, hi], -1).reshape(E, N, Kd)]
    w = words[: E * N * Kd // 32].copy().reshape(E, N // 128, Kd // 128, 128, 4)
    sbytes = w.transpose(0, 1, 3, 2, 4).reshape(E, N, Kd // 32).astype(np.int64)
    val = e2m1 * np.repeat(np.ldexp(1.0, sbytes - 127), 32, axis=-1)
    val = val * alpha.astype(np.float64)[:, None, None]
    out = np.empty((E, N, Kd))
    R = np.arange(N)
    if gated:
        b, t, r = R // 256, (R // 128) % 2, R % 128
        gate0, up0 = (0, I) if layout == 0 else (I, 0)
        src = np.where(t == 0, gate0, up0) + 128 * b + r
    else:
        src = R
    out[:, src, :] = val
    return out


def dequant_reference(codes_packed, scales, gran, gs):
    """Plain decode of raw [E, N, Kd/2] codes + [E, N, Kd/g] scales."""
    lo, hi = codes_packed & 0xF, codes_packed >> 4
    codes = np.stack([lo, hi], -1).reshape(*codes_packed.shape[:-1], -1)
    t = torch.from_numpy(np.ascontiguousarray(scales))
    if gran == 16:
        sv = t.view(torch.float8_e4m3fn).double().numpy()
    else:
        sv = t.view(torch.float8_e8m0fnu).double().numpy()
    return E2M1[codes] * np.repeat(sv, gran, axis=-1) * gs.astype(
        np.float64)[:, None, None]


# ------------------------------------------------- MoE two-level parity check
# The intermediate h = silu(G) * U is rounded (bf16, or E4M3 x UE8M0/32)
# between FC1 and FC2.  The GPU takes that decision from its FP32 value and
# the oracle from its FP64 value, so where the exact h sits closer to a
# rounding boundary than the FP32 error of G and U can reach, more than one
# code is a correct rounding (several results are correct).  The check
#  (1) compares the GPU's h (read back from the workspace) with the oracle's
#      rounded h.  They must be equal, except that the GPU's code may be a
#      correct rounding of another value within the FP32 error radius r of
#      the exact h: the adjacent code when h lies within r of the boundary
#      between the two, and a code further away only where r itself spans
#      more than one code (h near zero after cancellation in G or U); in the
#      FP8 path also the rounding under the neighbouring group exponent when
#      the group's maximum sits within its radius of an exponent boundary.
#      Such ties may be at most MAX_TIE_FRAC of all h elements;
#  (2) compares y with the oracle's y under the stated tolerance
#      |d| <= 2^-7 |ref| + 1e-3 rms(ref), widened for an output element only
#      by the exact effect of those tie choices, sum_j |w_j w2[c, i] dh_i|.
#
# The radius is a first-order bound on the FP32 error of G (and U) under a
# pessimistic model of the tensor core's accumulation: each K step adds 16
# exact products to the running sum S, aligning the 17 addends to the
# largest and truncating each (an error below u = 2^-23 of the largest,
# <= 17 u max(|S_{s-1}|, max|t|) <= 17 u (|S_{s-1}| + sum_step |t|)), then
# rounds the result (<= u |S_s|).  Summed over the steps:
#     |G_fp32 - G| <= u (18 sum_s |S_s| + 17 sum_k |t_k|),
# with S_s the running sums after each chunk of 16 and t_k the terms (the
# oracle returns both sums in FP64).  The radius takes twice that (other
# summation orders: partial accumulators summed in the epilogue, 32-wide
# K steps), propagates it through silu(G) * U to first order and adds
# 2^-17 |h| for the epilogue's elementwise FP32 operations (fast exponential
# and division).
#
# MAX_TIE_FRAC: a tie can only occur where the exact h lies within the
# GPU's error of a rounding boundary.  The bf16 boundaries are one ulp
# apart (relative spacing 2^-8 .. 2^-7), so a relative error delta in h gives
# a tie rate of about 2 delta / 2^-7.5 ~ 360 delta.  The highest rate seen on
# the GB300 is 1.31e-3 (the decode workload: 1378 of 1,048,576 h elements),
# i.e. delta ~ 3.6e-6 -- FP32 accumulation over 384 tensor-core K steps plus
# the fast SiLU.  The cap allows 2.3x that rate (delta up to ~8e-6); a
# systematic error of one ulp would flip half of all elements.
MAX_TIE_FRAC = 3e-3
RADIUS_MARGIN = 2.0
U32 = 2.0 ** -23


def _silu(g):
    return g / (1.0 + np.exp(-g))


def moe_radius(aux, K=None):
    """FP32 error radius of the GPU's h, per element (aux from the oracle)."""
    G, U = aux[..., 0], aux[..., 1]
    SG, SU, PG, PU = aux[..., 2], aux[..., 3], aux[..., 4], aux[..., 5]
    rG = RADIUS_MARGIN * U32 * (18.0 * PG + 17.0 * SG)
    rU = RADIUS_MARGIN * U32 * (18.0 * PU + 17.0 * SU)
    sig = 1.0 / (1.0 + np.exp(-G))
    dsilu = sig * (1.0 + G * (1.0 - sig))
    h = _silu(G) * U
    return np.abs(U * dsilu) * rG + np.abs(_silu(G)) * rU + 2.0 ** -17 * np.abs(h)


def _bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns of values that are exactly bf16."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.int64)


def _ordered(bits, sign_bit):
    """Sign-magnitude codes -> integers in value order (+0 and -0 both 0)."""
    mag = bits & (sign_bit - 1)
    return np.where(bits & sign_bit, -mag, mag)


def _bf16_of_ordered(o):
    """Inverse of _ordered for bf16: value of the code at order o."""
    bits = (0x8000 | -o) if o < 0 else o
    return float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0])


def _tie_bf16(orc, h, r, vg, vo):
    """(admissible, code distance, radius use) of the GPU code vg."""
    rnd = lambda v: orc.bf16_value(orc.bf16_rne(v))   # noqa: E731
    og, oo = (int(x) for x in _ordered(_bf16_bits([vg, vo]), 0x8000))
    dist = abs(og - oo)
    # distance from h to the values that round to vg
    lo = 0.5 * (vg + _bf16_of_ordered(og - 1))
    hi = 0.5 * (vg + _bf16_of_ordered(og + 1))
    gap = (lo - h) if h < lo else (h - hi) if h > hi else 0.0
    ok = rnd(h - r) <= vg <= rnd(h + r)
    return ok, dist, (gap / r if r > 0 else np.inf)


def _e4m3_ordered(c):
    return -(c & 0x7F) if c & 0x80 else (c & 0x7F)


def _e4m3_of_ordered(o):
    return (0x80 | -o) if o < 0 else o


def _tie_fp8(orc, hgrp, rgrp, idx, vg, vo):
    """(admissible, code distance, radius use) for one element of a group.

    Admissible: vg is the E4M3 rounding, under a group exponent that a
    maximum within the radius can select, of a value within r of h."""
    amax = float(np.abs(hgrp).max())
    rmax = float(rgrp[np.argmax(np.abs(hgrp))])
    lo = orc.fp8_group_exponent(np.full(32, max(amax - rmax, 0.0)))
    hi = orc.fp8_group_exponent(np.full(32, amax + rmax))
    h, r = float(hgrp[idx]), float(rgrp[idx])
    for e in range(lo, hi + 1):
        sc = 2.0 ** e

        def rnd(v, sc=sc):
            return orc.e4m3_value(orc.e4m3_rne_sat(v / sc)) * sc
        # vg must be a code under this exponent and within the rounded range
        if rnd(vg) != vg or not rnd(h - r) <= vg <= rnd(h + r):
            continue
        og = _e4m3_ordered(orc.e4m3_rne_sat(vg / sc))
        oh = _e4m3_ordered(orc.e4m3_rne_sat(h / sc))
        if og == oh:            # only the group exponent differs
            return True, 0, 0.0
        nb = orc.e4m3_value(_e4m3_of_ordered(og - 1 if og > oh else og + 1)) * sc
        use = abs(h - 0.5 * (vg + nb)) / r if r > 0 else np.inf
        return True, abs(og - oh), use
    return False, -1, np.inf


def w2_columns(w, e, cols, gran):
    """Dequantized FC2 weight columns w2[e][:, cols] (FP64, gs included)."""
    codes = w["w2"][e]                      # [K, I/2]
    scales = w["w2_s"][e]                   # [K, I/gran]
    out = []
    for i in cols:
        byte = codes[:, i // 2]
        c = (byte & 0xF) if i % 2 == 0 else (byte >> 4)
        t = torch.from_numpy(np.ascontiguousarray(scales[:, i // gran]))
        sv = (t.view(torch.float8_e4m3fn) if gran == 16 else
              t.view(torch.float8_e8m0fnu)).double().numpy()
        out.append(E2M1[c] * sv * float(w["w2_gs"][e]))
    return np.stack(out, 1) if out else np.zeros((codes.shape[0], 0))


def check_moe_values(orc, *, K, gran, act_mode, h_gpu, y_gpu, ref_y, ref_h,
                     aux, ids, wts, w_used, what, tie_frac=MAX_TIE_FRAC):
    """The two-level check on plain arrays.

    h_gpu [ntok, k, I]: the GPU's rounded h (FP64 of its exact values);
    y_gpu [ntok, K]: the GPU's y; ref_y, ref_h, aux: the oracle's unrounded
    y and h and its aux; ids, wts [ntok, k]: the oracle's routing of these
    tokens.  Raises AssertionError on a violation; returns the statistics
    (tie count and fraction, largest use of the radius by a tie, largest
    ratio of |error| to the allowed bound in y)."""
    h_gpu = np.asarray(h_gpu, dtype=np.float64)
    h_ref = orc.round_intermediate(ref_h, act_mode).reshape(h_gpu.shape)
    radius = moe_radius(aux)
    mism = np.argwhere(h_gpu != h_ref)
    stats = {"ties": int(len(mism)), "h_elements": int(h_ref.size),
             "tie_frac": len(mism) / max(h_ref.size, 1),
             "tie_cap": tie_frac, "max_tie_radius_use": 0.0,
             "multi_code_ties": 0, "max_code_distance": 0}
    assert len(mism) <= tie_frac * h_ref.size, (
        f"{what}: h differs from the oracle in {len(mism)} of {h_ref.size} "
        f"elements (cap {tie_frac:g})")
    allow = np.zeros(np.shape(ref_y))
    for n, j, i in mism:
        h, r = ref_h[n, j, i], radius[n, j, i]
        vo, vg = h_ref[n, j, i], h_gpu[n, j, i]
        if act_mode == 0:
            ok, dist, use = _tie_bf16(orc, h, r, vg, vo)
        else:
            g0 = (i // 32) * 32
            ok, dist, use = _tie_fp8(orc, ref_h[n, j, g0:g0 + 32],
                                     radius[n, j, g0:g0 + 32], i - g0, vg, vo)
        assert ok, (f"{what}: h[token {n}, slot {j}, {i}] = {vg!r} is not an "
                    f"admissible rounding of {h!r} (radius {r:.3g}, oracle "
                    f"{vo!r})")
        stats["max_tie_radius_use"] = max(stats["max_tie_radius_use"],
                                          float(use))
        stats["multi_code_ties"] += int(dist > 1)
        stats["max_code_distance"] = max(stats["max_code_distance"], dist)
        col = w2_columns(w_used, int(ids[n, j]), [int(i)], gran)[:, 0]
        allow[n] += np.abs(wts[n, j] * col * (vg - vo))
    _, err, bound, rms = tolerance_violations(y_gpu, ref_y)
    ratio = err / (bound + allow)
    stats["y_max_ratio"] = float(ratio.max()) if ratio.size else 0.0
    bad = ratio > 1.0
    if bad.any():
        idx = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} y elements outside "
            f"2^-7|ref| + 1e-3 rms (+ tie effect); {len(mism)} h ties; worst "
            f"at {idx}: gpu {y_gpu[idx]!r} ref {ref_y[idx]!r}")
    return stats


def read_h(fp4, packed, ws, T, k, I, tokens):
    """The GPU's rounded h rows of `tokens` [ntok, k, I] from the workspace
    (bf16 values, or E4M3 bytes times their UE8M0 group scales)."""
    offs = fp4.moe_workspace_offsets(packed, T, k)
    P = T * k
    inv = ws[offs["inv"]:offs["inv"] + 4 * P].view(torch.int32).cpu().numpy()
    rows = [int(inv[t * k + j]) for t in tokens for j in range(k)]
    ridx = torch.tensor(rows, device=ws.device)
    if offs["h_format"] == 0:
        hb = ws[offs["h"]:offs["h"] + 2 * P * I].view(torch.int16).view(
            torch.bfloat16).view(P, I)
        h = hb[ridx].float().cpu().numpy().astype(np.float64)
    else:
        pitch = offs["pitch"]
        h8 = ws[offs["h"]:offs["h"] + P * I].view(P, I)[ridx].cpu()
        q = h8.view(torch.float8_e4m3fn).double().numpy()
        hs = ws[offs["h_scales"]:offs["h_scales"] + (I // 128) * pitch * 4]
        hs = hs.view(I // 128, pitch, 4).cpu().numpy()
        sb = hs[:, rows, :].transpose(1, 0, 2).reshape(len(rows), I // 32)
        h = q * np.repeat(np.ldexp(1.0, sb.astype(np.int64) - 127), 32, axis=-1)
    return h.reshape(len(tokens), k, I)


def check_moe(orc, fp4, cfg, packed, y, ws, tokens, ref_y, ref_h, ref_aux,
              w_used, gran, act_mode, logits, what, record=None):
    tokens = list(tokens)
    h_gpu = read_h(fp4, packed, ws, cfg.T, cfg.top_k, cfg.I, tokens)
    ids, wts = orc.route(logits[tokens], cfg.top_k)
    y_gpu = to_f64(y[tokens]) if isinstance(y, torch.Tensor) else y
    stats = check_moe_values(
        orc, K=cfg.K, gran=gran, act_mode=act_mode, h_gpu=h_gpu, y_gpu=y_gpu,
        ref_y=ref_y, ref_h=ref_h.reshape(h_gpu.shape), aux=ref_aux, ids=ids,
        wts=wts, w_used=w_used, what=what)
    if record is not None:
        for key, v in stats.items():
            record(key, v)
    print(f"{what}: {stats}")
    return stats
