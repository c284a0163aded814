"""Pins for the FP64 oracle, checked against things other than itself.

The pages print no worked example, so each pin is a closed form, an
invariant, a library routine (PyTorch's float8 / bfloat16 conversions, numpy
FP64 matmul, scipy softmax) or brute force with exact rationals.  Each pin is
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign,
a swapped nibble, a transposed operand, a wrong tie rule) fails it.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E2M1_MAG = [Fr(0), Fr(1, 2), Fr(1), Fr(3, 2), Fr(2), Fr(3), Fr(4), Fr(6)]
E2M1_SIGNED = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3,
                        -4, -6])


def torch_e4m3(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).double().numpy()


def torch_ue8m0(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8))
    return t.view(torch.float8_e8m0fnu).double().numpy()


# ------------------------------------------------------------------ codecs

def test_e2m1_codebook_and_roundtrip(orc):
    # The codebook {0,0.5,1,1.5,2,3,4,6} with a sign bit.
    for c in range(16):
        v = orc.e2m1_value(c)
        assert v == E2M1_SIGNED[c]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)
        assert orc.e2m1_rne(v) == c            # all 16 codes round-trip


@pytest.mark.parametrize("v,code", [
    (0.25, 0x0), (0.2500001, 0x1), (0.75, 0x2), (0.7499999, 0x1),
    (1.25, 0x2), (1.2500001, 0x3), (1.75, 0x4), (2.5, 0x4), (2.5000001, 0x5),
    (3.5, 0x6), (3.4999999, 0x5), (5.0, 0x6), (5.0000001, 0x7), (6.0, 0x7),
    (7.0, 0x7), (1e9, 0x7), (-0.25, 0x8), (-0.0, 0x8), (-0.1, 0x8),
    (-5.0, 0xE), (-2.5, 0xC), (0.0, 0x0)])
def test_e2m1_rne_ties(orc, v, code):
    # Ties go to the even mantissa bit: 0.25->0, 0.75->1, 1.25->1, 1.75->2,
    # 2.5->2, 3.5->4, 5->4; |v| > 6 saturates; the sign of zero is kept.
    assert orc.e2m1_rne(v) == code


def test_e4m3_decode_matches_torch_all_bytes(orc):
    ref = torch_e4m3(np.arange(256))
    for b in range(256):
        v = orc.e4m3_value(b)
        if b in (0x7F, 0xFF):
            assert math.isnan(v) and math.isnan(ref[b])
        else:
            assert v == ref[b], hex(b)
    assert orc.e4m3_value(0x7E) == 448.0
    assert orc.e4m3_value(0x01) == 2.0 ** -9
    assert orc.e4m3_value(0x38) == 1.0


def test_e4m3_roundtrip_all_finite(orc):
    n = 0
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert orc.e4m3_rne_sat(orc.e4m3_value(b)) == b, hex(b)
        n += 1
    assert n == 254


def test_e4m3_rne_matches_torch(orc):
    g = np.random.default_rng(7)
    v = np.concatenate([
        g.standard_normal(4000) * 10.0 ** g.uniform(-4, 2.5, 4000),
        # exact midpoints between neighbouring codes (ties)
        (torch_e4m3(np.arange(1, 126)) + torch_e4m3(np.arange(2, 127))) / 2,
        -(torch_e4m3(np.arange(1, 126)) + torch_e4m3(np.arange(2, 127))) / 2,
    ])
    v = v[np.abs(v) < 464.0].astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_rne_sat(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)
    assert orc.e4m3_rne_sat(1e6) == 0x7E and orc.e4m3_rne_sat(-500) == 0xFE


def test_ue8m0_decode_matches_torch(orc):
    ref = torch_ue8m0(np.arange(256))
    for b in range(255):
        assert orc.ue8m0_value(b) == ref[b] == 2.0 ** (b - 127)
    assert math.isnan(orc.ue8m0_value(255))


def test_bf16_rne_matches_torch(orc):
    g = np.random.default_rng(11)
    v = np.concatenate([
        g.standard_normal(5000) * 10.0 ** g.uniform(-40, 38, 5000),
        # float32 values exactly half-way between bf16 neighbours
        ((g.integers(0, 2**15, 2000).astype(np.uint32) << 16) | 0x8000)
        .view(np.float32).astype(np.float64),
    ]).astype(np.float32)
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy()
    got = np.array([orc.bf16_rne(float(x)) for x in v], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref.view(np.uint16))
    for bits in (0x0001, 0x3F80, 0xC2F7, 0x7F7F, 0x8000):
        assert orc.bf16_value(bits) == float(
            torch.tensor([bits], dtype=torch.int32).to(torch.int16)
            .view(torch.bfloat16).float())


# ------------------------------------------------------------------ requant

def _brute_group(codes, sbytes):
    """Exact rational requant of one 32-group (independent of the oracle)."""
    svals = torch_e4m3(np.array(sbytes))
    if any(math.isnan(s) for s in svals):
        return [0] * 32, 0xFF
    vals, signs = [], []
    for i, c in enumerate(codes):
        sb = sbytes[i // 16]
        mag = E2M1_MAG[c & 7] * Fr(abs(svals[i // 16]))
        vals.append(mag)
        signs.append(bool(c & 8) != bool(sb & 0x80))
    amax = max(vals)
    if amax == 0:
        e = 0
    else:
        e = next(e for e in range(-60, 60) if 6 * Fr(2) ** e >= amax)
    byte = min(254, max(0, e + 127))
    scale = Fr(2) ** (byte - 127)
    out = []
    for m, s in zip(vals, signs):
        y = m / scale
        best = min(range(8), key=lambda c: (abs(y - E2M1_MAG[c]), c & 1))
        out.append(best | (8 if s else 0))
    return out, byte


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8).reshape(-1, 2)
    return (codes[:, 0] | (codes[:, 1] << 4)).astype(np.uint8)


def test_requant_brute_force(orc):
    g = np.random.default_rng(5)
    finite = np.array([b for b in range(256) if b not in (0x7F, 0xFF)],
                      dtype=np.uint8)
    rows, K = 40, 96
    codes = g.integers(0, 16, size=(rows, K), dtype=np.uint8)
    s16 = g.choice(finite, size=(rows, K // 16))
    # a few structured rows: a zero group, a NaN scale, huge/tiny halves
    s16[0, :2] = 0
    s16[1, 2] = 0x7F
    s16[2, 0], s16[2, 1] = 0x7E, 0x01
    packed = np.stack([_pack(r) for r in codes])
    out, s32 = orc.requant(packed, s16)
    for r in range(rows):
        for gi in range(K // 32):
            ref_codes, ref_byte = _brute_group(
                codes[r, gi * 32:(gi + 1) * 32], s16[r, gi * 2:gi * 2 + 2])
            assert s32[r, gi] == ref_byte
            np.testing.assert_array_equal(
                out[r, gi * 16:(gi + 1) * 16], _pack(ref_codes))


def test_requant_idempotent_on_group32_exact(orc):
    # Both halves share scale 2^e and the largest magnitude is 4 or 6: the
    # recomputed UE8M0 scale is 2^e and every code comes back unchanged.
    g = np.random.default_rng(9)
    rows, K = 64, 256
    codes = g.integers(0, 16, size=(rows, K), dtype=np.uint8)
    e = g.integers(-6, 9, size=(rows, K // 32))
    top = g.choice([0x6, 0x7, 0xE, 0xF], size=(rows, K // 32))
    for r in range(rows):
        for gi in range(K // 32):
            grp = codes[r, gi * 32:(gi + 1) * 32]
            grp[np.isin(grp & 7, [6, 7])] &= 0xD   # keep magnitudes < 4 ...
            grp[g.integers(0, 32)] = top[r, gi]    # ... except one 4 or 6
    s16 = np.repeat(((e + 7) << 3).astype(np.uint8), 2, axis=1)
    packed = np.stack([_pack(r) for r in codes])
    out, s32 = orc.requant(packed, s16)
    np.testing.assert_array_equal(out, packed)
    np.testing.assert_array_equal(s32, (e + 127).astype(np.uint8))


def test_requant_smaller_max_keeps_values(orc):
    # Max magnitude 3 with scale 2^e: the new scale is 2^(e-1) and every value
    # {0.5,1,1.5,3}*2^e doubles onto the grid exactly -- same values, new codes.
    g = np.random.default_rng(3)
    mags = np.array([0, 1, 2, 3, 5], dtype=np.uint8)
    codes = g.choice(mags, size=(8, 64)) | (g.integers(0, 2, (8, 64)) << 3)
    codes[:, 0] = 5
    codes[:, 32] = 5
    codes = codes.astype(np.uint8)
    s16 = np.full((8, 4), (2 + 7) << 3, dtype=np.uint8)     # 2^2
    out, s32 = orc.requant(np.stack([_pack(r) for r in codes]), s16)
    assert (s32 == 127 + 1).all()
    lo, hi = out & 0xF, out >> 4
    new = np.stack([lo, hi], -1).reshape(8, 64)
    np.testing.assert_array_equal(E2M1_SIGNED[new] * 2.0,
                                  E2M1_SIGNED[codes] * 4.0)


def test_requant_hand_examples(orc):
    # tests/golden/requant_hand_examples.txt: worked by hand from the
    # requantization rule (the notes page, "Requantization path": dequantize
    # with the group16 scales, recompute a group32 scale, round to E2M1).
    path = os.path.join(GOLDEN, "requant_hand_examples.txt")
    cases = []
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                cases.append([int(t, 16) for t in line.split()])
    assert len(cases) >= 3
    for c in cases:
        s_lo, s_hi, c_lo, c_hi, want_byte, want_lo, want_hi = c
        codes = np.array([c_lo] * 16 + [c_hi] * 16, dtype=np.uint8)
        out, s32 = orc.requant(_pack(codes)[None, :],
                               np.array([[s_lo, s_hi]], dtype=np.uint8))
        assert s32[0, 0] == want_byte
        assert out[0, 0] == (want_lo | (want_lo << 4))
        assert out[0, 15] == (want_hi | (want_hi << 4))


def test_requant_rejects_ragged_k(orc):
    with pytest.raises(ValueError):
        orc.requant(np.zeros((2, 8), np.uint8), np.zeros((2, 1), np.uint8))


# ------------------------------------------------------------------ routing

def _softmax(x):
    x = x - x.max(axis=-1, keepdims=True)
    p = np.exp(x)
    return p / p.sum(axis=-1, keepdims=True)


def test_route_against_numpy_softmax(orc):
    g = np.random.default_rng(1)
    logits = g.standard_normal((300, 64)).astype(np.float32)
    ids, w = orc.route(logits, 6)
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :6]
    np.testing.assert_array_equal(ids, order)
    full = _softmax(logits.astype(np.float64))
    sel = np.take_along_axis(full, ids, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)


def test_route_k_equals_e_is_softmax(orc):
    import scipy.special
    g = np.random.default_rng(2)
    logits = g.standard_normal((20, 16)).astype(np.float32)
    ids, w = orc.route(logits, 16)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids, 1), rtol=1e-13)


def test_route_ties_go_to_lower_id(orc):
    logits = np.zeros((2, 8), dtype=np.float32)
    logits[0, [5, 2, 7]] = 1.0
    logits[1, :] = -3.0
    ids, w = orc.route(logits, 4)
    assert list(ids[0]) == [2, 5, 7, 0]
    assert list(ids[1]) == [0, 1, 2, 3]
    np.testing.assert_allclose(w[1], 0.25, rtol=1e-15)


def test_route_rejects_nan(orc):
    logits = np.zeros((1, 4), dtype=np.float32)
    logits[0, 1] = np.nan
    with pytest.raises(ValueError):
        orc.route(logits, 2)


def test_permute_invariants(orc):
    g = np.random.default_rng(4)
    T, k, E = 257, 3, 11
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(
        np.int32)
    counts, offsets, perm, inv = orc.permute(ids, E)
    flat = ids.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert (np.diff(offsets) == counts).all()
    np.testing.assert_array_equal(np.sort(perm), np.arange(T * k))
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()          # stable: ascending pair index
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))


# ------------------------------------------------------------------ act quant

def test_act_quant_against_torch(orc):
    g = np.random.default_rng(6)
    x = g.standard_normal((9, 128)).astype(np.float32)
    x[0] *= 1e-20
    x[1] *= 1e4
    x[2, :32] = 0
    xb = synth.f32_to_bf16_bits(x)
    q, s = orc.act_quant(xb)
    xv = synth.bf16_bits_to_f32(xb).astype(np.float64).reshape(9, 4, 32)
    amax = np.abs(xv).max(-1)
    for t in range(9):
        for gi in range(4):
            b = int(s[t, gi])
            if amax[t, gi] == 0:
                assert b == 127
                continue
            e = b - 127
            assert amax[t, gi] <= 448 * 2.0 ** e
            assert amax[t, gi] > 448 * 2.0 ** (e - 1)
            ref = torch.from_numpy((xv[t, gi] / 2.0 ** e).astype(np.float32)).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(q[t, gi * 32:(gi + 1) * 32], ref)


# ------------------------------------------------------------------ MoE

def _dequant(codes_packed, scales, gran, gs):
    """Independent numpy decode: [E, N, Kd/2] + [E, N, Kd/g] -> [E, N, Kd]."""
    lo, hi = codes_packed & 0xF, codes_packed >> 4
    codes = np.stack([lo, hi], -1).reshape(*codes_packed.shape[:-1], -1)
    sv = torch_e4m3(scales) if gran == 16 else torch_ue8m0(scales)
    return (E2M1_SIGNED[codes] * np.repeat(sv, gran, axis=-1)
            * gs.astype(np.float64)[:, None, None])


def _dense_reference(x, W13, W2, w13_layout, act_mode, I):
    gate = W13[:I] if w13_layout == 0 else W13[I:]
    up = W13[I:] if w13_layout == 0 else W13[:I]
    G = gate @ x
    U = up @ x
    h = G / (1 + np.exp(-G)) * U
    if act_mode == 0:
        h = torch.from_numpy(h).to(torch.bfloat16).double().numpy()
    else:
        hg = h.reshape(-1, 32)
        out = np.empty_like(hg)
        for i, grp in enumerate(hg):
            a = np.abs(grp).max()
            e = 0 if a == 0 else math.ceil(math.log2(a / 448))
            while 448 * 2.0 ** e < a:
                e += 1
            while a > 0 and 448 * 2.0 ** (e - 1) >= a:
                e -= 1
            q = torch.from_numpy((grp / 2.0 ** e).astype(np.float32)).to(
                torch.float8_e4m3fn).double().numpy()
            out[i] = q * 2.0 ** e
        h = out.reshape(-1)
    return W2 @ h


def _tiny_weights(E, K, I, seed, gran=16):
    cfg = synth.MoeConfig("pin", E, K, I, 4, 1, weight_seed=seed)
    w = synth.moe_weights(cfg, threads=2)
    return w


@pytest.mark.parametrize("w13_layout", [0, 1])
def test_moe_one_expert_top1_is_dense_gemm(orc, w13_layout):
    E, K, I, T = 1, 96, 64, 5
    w = _tiny_weights(E, K, I, 41)
    g = np.random.default_rng(8)
    xb = synth.f32_to_bf16_bits(g.standard_normal((T, K)).astype(np.float32))
    logits = g.standard_normal((T, E)).astype(np.float32)
    y = orc.moe_rows(range(T), **w, gran=16, w13_layout=w13_layout,
                     act_mode=0, top_k=1, logits=logits, x_bf16=xb)
    W13 = _dequant(w["w13"], w["w13_s"], 16, w["w13_gs"])[0]
    W2 = _dequant(w["w2"], w["w2_s"], 16, w["w2_gs"])[0]
    xv = synth.bf16_bits_to_f32(xb).astype(np.float64)
    for t in range(T):
        ref = _dense_reference(xv[t], W13, W2, w13_layout, 0, I)
        np.testing.assert_allclose(y[t], ref, rtol=1e-9,
                                   atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("gran", [32, 16])
def test_moe_fp8_one_expert_top1_is_dense_gemm(orc, gran):
    E, K, I, T = 1, 64, 96, 4
    w = _tiny_weights(E, K, I, 42)
    if gran == 32:
        # group32 UE8M0 weights, as the FP8 path consumes them after requant
        w13 = w["w13"].reshape(-1, K // 2)
        w13q, w13s = orc.requant(w13, w["w13_s"].reshape(-1, K // 16))
        w2q, w2s = orc.requant(w["w2"].reshape(-1, I // 2),
                               w["w2_s"].reshape(-1, I // 16))
        wg = dict(w13=w13q.reshape(w["w13"].shape),
                  w13_s=w13s.reshape(E, 2 * I, K // 32), w13_gs=w["w13_gs"],
                  w2=w2q.reshape(w["w2"].shape), w2_s=w2s.reshape(E, K, I // 32),
                  w2_gs=w["w2_gs"])
    else:
        wg = w   # group16 weights kept under FP8 activations
    g = np.random.default_rng(10)
    xb = synth.f32_to_bf16_bits(g.standard_normal((T, K)).astype(np.float32))
    xq, xs = orc.act_quant(xb)
    logits = g.standard_normal((T, E)).astype(np.float32)
    y = orc.moe_rows(range(T), **wg, gran=gran, w13_layout=0, act_mode=1,
                     top_k=1, logits=logits, xq=xq, xs=xs)
    W13 = _dequant(wg["w13"], wg["w13_s"], gran, w["w13_gs"])[0]
    W2 = _dequant(wg["w2"], wg["w2_s"], gran, w["w2_gs"])[0]
    xv = torch_e4m3(xq) * np.repeat(torch_ue8m0(xs), 32, axis=1)
    for t in range(T):
        ref = _dense_reference(xv[t], W13, W2, 0, 1, I)
        np.testing.assert_allclose(y[t], ref, rtol=1e-9,
                                   atol=1e-12 * np.abs(ref).max())


def test_moe_identical_experts_independent_of_routing(orc):
    E, K, I, T = 6, 64, 32, 3
    w = _tiny_weights(1, K, I, 43)
    rep = {k: np.repeat(v, E, axis=0) for k, v in w.items()}
    g = np.random.default_rng(12)
    xb = synth.f32_to_bf16_bits(g.standard_normal((T, K)).astype(np.float32))
    l1 = g.standard_normal((T, E)).astype(np.float32)
    l2 = g.standard_normal((T, E)).astype(np.float32)
    common = dict(gran=16, w13_layout=0, act_mode=0, x_bf16=xb)
    y1 = orc.moe_rows(range(T), **rep, top_k=3, logits=l1, **common)
    y2 = orc.moe_rows(range(T), **rep, top_k=2, logits=l2, **common)
    y0 = orc.moe_rows(range(T), **w, top_k=1,
                      logits=np.zeros((T, 1), np.float32), **common)
    np.testing.assert_allclose(y1, y0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(y2, y0, rtol=1e-13, atol=1e-15)


def test_moe_brute_force_tiny(orc):
    # Pure-Python loops, one multiply-add at a time, on a 3-expert top-2 layer.
    E, K, I, T, k = 3, 32, 32, 2, 2
    w = _tiny_weights(E, K, I, 44)
    g = np.random.default_rng(13)
    xb = synth.f32_to_bf16_bits(g.standard_normal((T, K)).astype(np.float32))
    logits = g.standard_normal((T, E)).astype(np.float32)
    y = orc.moe_rows(range(T), **w, gran=16, w13_layout=1, act_mode=0,
                     top_k=k, logits=logits, x_bf16=xb)

    def wv(codes, scales, gs, e, row, col):
        byte = int(codes[e, row, col // 2])
        c = byte & 0xF if col % 2 == 0 else byte >> 4
        s = float(torch_e4m3(np.array([scales[e, row, col // 16]]))[0])
        return float(E2M1_SIGNED[c]) * s * float(gs[e])

    xv = synth.bf16_bits_to_f32(xb).astype(np.float64)
    for t in range(T):
        lg = [float(v) for v in logits[t]]
        chosen = sorted(range(E), key=lambda e: (-lg[e], e))[:k]
        ex = [math.exp(lg[e] - lg[chosen[0]]) for e in chosen]
        ref = [0.0] * K
        for j, e in enumerate(chosen):
            h = []
            for i in range(I):
                up = sum(xv[t, c] * wv(w["w13"], w["w13_s"], w["w13_gs"], e, i, c)
                         for c in range(K))
                gt = sum(xv[t, c] * wv(w["w13"], w["w13_s"], w["w13_gs"], e,
                                       I + i, c) for c in range(K))
                hv = gt / (1 + math.exp(-gt)) * up
                h.append(float(torch.tensor(hv, dtype=torch.float64)
                               .to(torch.bfloat16).double()))
            for n in range(K):
                o = sum(h[i] * wv(w["w2"], w["w2_s"], w["w2_gs"], e, n, i)
                        for i in range(I))
                ref[n] += ex[j] / sum(ex) * o
        np.testing.assert_allclose(y[t], ref, rtol=1e-9,
                                   atol=1e-12 * max(map(abs, ref)))


def test_moe_layout_flag_swaps_halves(orc):
    E, K, I, T = 4, 64, 32, 6
    w = _tiny_weights(E, K, I, 45)
    g = np.random.default_rng(14)
    xb = synth.f32_to_bf16_bits(g.standard_normal((T, K)).astype(np.float32))
    logits = g.standard_normal((T, E)).astype(np.float32)
    swapped = dict(w)
    swapped["w13"] = np.concatenate([w["w13"][:, I:], w["w13"][:, :I]], 1)
    swapped["w13_s"] = np.concatenate([w["w13_s"][:, I:], w["w13_s"][:, :I]], 1)
    a = orc.moe_rows(range(T), **w, gran=16, w13_layout=0, act_mode=0,
                     top_k=2, logits=logits, x_bf16=xb)
    b = orc.moe_rows(range(T), **swapped, gran=16, w13_layout=1, act_mode=0,
                     top_k=2, logits=logits, x_bf16=xb)
    np.testing.assert_array_equal(a, b)
