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
BIT_POS = [[6, 7, 8, 15], [22, 23, 24, 31], [3, 4, 5, 12], [19, 20, 21, 28],
           [0, 1, 2, 9], [16, 17, 18, 25], [14, 10, 11, 13], [30, 26, 27, 29]]
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
# the oracle from its FP64 value; where the two can straddle a rounding
# boundary both codes are correct.  The check therefore
#  (1) compares the GPU's h (read back from the workspace) with the oracle's
#      rounded h: equal everywhere, except where the GPU's code is a correct
#      rounding of some value within the FP32 error radius of the exact h;
#  (2) compares y with the oracle's y under the stated tolerance, widened for
#      an output element only by the exact effect of those tie choices.
# The radius bounds FP32 accumulation over K terms in any order with at most
# one ulp per operation (Higham's gamma_K with u = 2^-23) and propagates it
# through silu(G) * U, plus 2^-17 |h| for the elementwise FP32 operations
# (the epilogue's fast exponential and division are accurate to a few ulp
# over the range of G that occurs).

MAX_TIE_FRAC = 0.01


def _silu(g):
    return g / (1.0 + np.exp(-g))


def _radius(aux, K):
    G, U, SG, SU = aux[..., 0], aux[..., 1], aux[..., 2], aux[..., 3]
    gamma = K * 2.0 ** -23
    sig = 1.0 / (1.0 + np.exp(-G))
    dsilu = sig * (1.0 + G * (1.0 - sig))
    h = _silu(G) * U
    return (np.abs(U * dsilu) * gamma * SG + np.abs(_silu(G)) * gamma * SU
            + 2.0 ** -17 * np.abs(h))


def _bf16_round(v: float) -> float:
    return float(torch.tensor(v, dtype=torch.float64).to(torch.float32)
                 .to(torch.bfloat16).double())


def _bf16_ok(h, r, vg) -> bool:
    return _bf16_round(h - r) <= vg <= _bf16_round(h + r) or \
        _bf16_round(h + r) <= vg <= _bf16_round(h - r)


def _fp8_ok(orc, hgroup, rgroup, idx, vg) -> bool:
    amax = float(np.abs(hgroup).max())
    rmax = float(rgroup.max())
    lo = orc.fp8_group_exponent(np.full(32, max(amax - rmax, 0.0)))
    hi = orc.fp8_group_exponent(np.full(32, amax + rmax))
    h, r = float(hgroup[idx]), float(rgroup[idx])
    for e in range(lo, hi + 1):
        a = orc.e4m3_value(orc.e4m3_rne_sat((h - r) / 2.0 ** e)) * 2.0 ** e
        b = orc.e4m3_value(orc.e4m3_rne_sat((h + r) / 2.0 ** e)) * 2.0 ** e
        if min(a, b) <= vg <= max(a, b):
            return True
    return False


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


def check_moe(orc, fp4, cfg, packed, y, ws, tokens, ref_y, ref_h, ref_aux,
              w_used, gran, act_mode, logits, what):
    tokens = list(tokens)
    k, I, T = cfg.top_k, cfg.I, cfg.T
    offs = fp4.moe_workspace_offsets(packed, T, k)
    P = T * k
    inv = ws[offs["inv"]:offs["inv"] + 4 * P].view(torch.int32).cpu().numpy()
    hb = ws[offs["h"]:offs["h"] + 2 * P * I].view(torch.int16).view(
        torch.bfloat16).view(P, I)
    rows = [int(inv[t * k + j]) for t in tokens for j in range(k)]
    h_gpu = hb[torch.tensor(rows, device=hb.device)].float().cpu().numpy()
    h_gpu = h_gpu.astype(np.float64).reshape(len(tokens), k, I)
    h_ref = orc.round_intermediate(ref_h, act_mode).reshape(len(tokens), k, I)
    radius = _radius(ref_aux, cfg.K)
    mism = np.argwhere(h_gpu != h_ref)
    assert len(mism) <= MAX_TIE_FRAC * h_ref.size, (
        f"{what}: h differs from the oracle in {len(mism)} of {h_ref.size}")
    ids, wts = orc.route(logits[tokens], k)
    allow = np.zeros((len(tokens), cfg.K))
    for n, j, i in mism:
        h, r = ref_h[n, j, i], radius[n, j, i]
        vo, vg = h_ref[n, j, i], h_gpu[n, j, i]
        if act_mode == 0:
            ok = _bf16_ok(h, r, vg)
        else:
            g0 = (i // 32) * 32
            ok = _fp8_ok(orc, ref_h[n, j, g0:g0 + 32],
                         radius[n, j, g0:g0 + 32], i - g0, vg)
        assert ok, (f"{what}: h[token {tokens[n]}, slot {j}, {i}] = {vg!r} is "
                    f"not a rounding of {h!r} +- {r:.3g} (oracle {vo!r})")
        col = w2_columns(w_used, int(ids[n, j]), [int(i)], gran)[:, 0]
        allow[n] += np.abs(wts[n, j] * col * (vg - vo))
    gpu = to_f64(y[tokens]) if isinstance(y, torch.Tensor) else y
    _, err, bound, rms = tolerance_violations(gpu, ref_y)
    bad = err > bound + allow
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound - allow), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} y elements outside "
            f"2^-7|ref| + 1e-3 rms (+ tie effect); {len(mism)} h ties; worst "
            f"at {idx}: gpu {gpu[idx]!r} ref {ref_y[idx]!r}")
    return len(mism)
