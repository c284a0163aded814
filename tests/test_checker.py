"""The MoE parity checker rejects wrong results (CPU only).

The GPU tests accept a differing intermediate h only where it is a correct
rounding of a value within the FP32 error radius of the exact h (in practice
the adjacent code, with h next to the boundary between the two), and widen
the y tolerance only by the exact effect of such ties.  These tests feed the checker the oracle's own result
(which must pass) and copies of it with planted mistakes (each must fail):
h two ulps off, a tie far from any boundary, too many ties, one expert's FC2
output scaled by 1.01, two token rows swapped, and an FP8 code two steps off.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest

import _util
import synth
from _util import check_moe_values, dequant_reference, requant_weights_oracle

SMALL_FP8 = synth.MoeConfig("checker_fp8_E8_K256_I128_T20_k2", 8, 256, 128,
                            20, 2, act="fp8", weight_seed=7101,
                            input_seed=7201)


@functools.lru_cache(maxsize=4)
def _case(cfg):
    import oracle as orc
    orc.build()
    w = synth.moe_weights(cfg)
    acts = synth.moe_activations(cfg)
    toks = list(range(cfg.T))
    if cfg.act == "fp8":
        w = requant_weights_oracle(orc, w, cfg.E, cfg.K, cfg.I)
        xq, xs = orc.act_quant(acts["x_bf16"])
        ref_y, ref_h, aux = orc.moe_rows(
            toks, **w, gran=32, w13_layout=0, act_mode=1, top_k=cfg.top_k,
            logits=acts["logits"], xq=xq, xs=xs, return_h=True)
        gran, act = 32, 1
    else:
        ref_y, ref_h, aux = orc.moe_rows(
            toks, **w, gran=16, w13_layout=0, act_mode=0, top_k=cfg.top_k,
            logits=acts["logits"], x_bf16=acts["x_bf16"], return_h=True)
        gran, act = 16, 0
    ids, wts = orc.route(acts["logits"], cfg.top_k)
    w2 = dequant_reference(w["w2"], w["w2_s"], gran, w["w2_gs"])  # [E, K, I]
    return dict(orc=orc, cfg=cfg, w=w, ref_y=ref_y, ref_h=ref_h, aux=aux,
                ids=ids, wts=wts, gran=gran, act=act, w2=w2,
                h_round=orc.round_intermediate(ref_h, act))


def _bf16_values(orc, v):
    bits = orc.bf16_rne_array(v).astype(np.uint32) << np.uint32(16)
    return bits.view(np.float32).astype(np.float64)


def _y_from_h(c, h, scale_expert=None, factor=1.0):
    """y as a correct GPU would produce it from the rounded h it chose."""
    y = np.zeros_like(c["ref_y"])
    for n in range(h.shape[0]):
        for j in range(h.shape[1]):
            e = int(c["ids"][n, j])
            o = c["w2"][e] @ h[n, j]
            if e == scale_expert:
                o = o * factor
            y[n] += c["wts"][n, j] * o
    return _bf16_values(c["orc"], y)


def _check(c, h, y, **kw):
    return check_moe_values(
        c["orc"], K=c["cfg"].K, gran=c["gran"], act_mode=c["act"], h_gpu=h,
        y_gpu=y, ref_y=c["ref_y"], ref_h=c["ref_h"], aux=c["aux"],
        ids=c["ids"], wts=c["wts"], w_used=c["w"], what="planted", **kw)


def _bf16_step(v, steps):
    """v moved by `steps` bf16 ulps away from zero (v exactly bf16)."""
    b = (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.int64)
    b = b + steps
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(
        np.float64)


def _pick(h, frac, seed):
    g = np.random.default_rng(seed)
    nz = np.argwhere(h != 0)
    n = max(1, int(round(frac * h.size)))
    return nz[g.choice(len(nz), size=n, replace=False)]


def _closest_to_boundary(c):
    """(index, adjacent code value) of the h element nearest a bf16
    rounding boundary, relative to its radius."""
    h, hr = c["ref_h"], c["h_round"]
    up, dn = _bf16_step(hr, 1), _bf16_step(hr, -1)
    dist = np.minimum(np.abs(h - 0.5 * (hr + up)), np.abs(h - 0.5 * (hr + dn)))
    r = _util.moe_radius(c["aux"], c["cfg"].K)
    idx = np.unravel_index(np.argmin(np.where(hr != 0, dist / r, np.inf)),
                           h.shape)
    nb = up[idx] if (abs(h[idx] - 0.5 * (hr[idx] + up[idx])) <
                     abs(h[idx] - 0.5 * (hr[idx] + dn[idx]))) else dn[idx]
    return idx, nb, float(dist[idx] / r[idx])


# --------------------------------------------------------------- accepted

@pytest.mark.parametrize("cfg", [synth.TINY, SMALL_FP8], ids=["bf16", "fp8"])
def test_oracle_result_passes(cfg):
    c = _case(cfg)
    h = c["h_round"].copy()
    st = _check(c, h, _y_from_h(c, h))
    assert st["ties"] == 0 and st["y_max_ratio"] <= 1.0


def test_tie_at_a_boundary_is_accepted():
    c = _case(synth.TINY)
    idx, nb, use = _closest_to_boundary(c)
    assert use <= 1.0, "the tiny workload has an h this close to a boundary"
    h = c["h_round"].copy()
    h[idx] = nb
    st = _check(c, h, _y_from_h(c, h))
    assert st["ties"] == 1 and st["max_tie_radius_use"] <= 1.0


# --------------------------------------------------------------- rejected

def test_rejects_h_two_ulps_off_on_2_percent():
    c = _case(synth.TINY)
    h = c["h_round"].copy()
    for n, j, i in _pick(h, 0.02, 1):
        h[n, j, i] = _bf16_step(h[n, j, i], 2)
    with pytest.raises(AssertionError):
        _check(c, h, _y_from_h(c, h))


def test_rejects_h_two_ulps_off_below_the_tie_cap():
    # three elements only: under the cap, so the radius alone must catch it
    c = _case(synth.TINY)
    h = c["h_round"].copy()
    for n, j, i in _pick(h, 3 / h.size, 2):
        h[n, j, i] = _bf16_step(h[n, j, i], 2)
    with pytest.raises(AssertionError, match="admissible"):
        _check(c, h, _y_from_h(c, h))


def test_rejects_adjacent_code_far_from_a_boundary():
    c = _case(synth.TINY)
    h, hr = c["ref_h"], c["h_round"]
    r = _util.moe_radius(c["aux"], c["cfg"].K)
    up = _bf16_step(hr, 1)
    far = np.abs(h - 0.5 * (hr + up)) / r
    idx = np.unravel_index(np.argmax(np.where(hr != 0, far, -1)), h.shape)
    assert far[idx] > 10
    hg = hr.copy()
    hg[idx] = up[idx]
    with pytest.raises(AssertionError, match="admissible"):
        _check(c, hg, _y_from_h(c, hg))


def test_rejects_too_many_ties(monkeypatch):
    # Every adjacent flip made admissible by an inflated radius: the cap on
    # the number of ties must still reject 2% of h flipped.
    c = _case(synth.TINY)
    monkeypatch.setattr(_util, "RADIUS_MARGIN", 1e9)
    h = c["h_round"].copy()
    for n, j, i in _pick(h, 0.02, 3):
        h[n, j, i] = _bf16_step(h[n, j, i], 1)
    with pytest.raises(AssertionError, match="cap"):
        _check(c, h, _y_from_h(c, h))


@pytest.mark.parametrize("cfg", [synth.TINY, SMALL_FP8], ids=["bf16", "fp8"])
def test_rejects_one_expert_fc2_scaled_by_1_01(cfg):
    c = _case(cfg)
    h = c["h_round"].copy()
    e = int(np.bincount(c["ids"].ravel()).argmax())
    y = _y_from_h(c, h, scale_expert=e, factor=1.01)
    with pytest.raises(AssertionError, match="y elements"):
        _check(c, h, y)


@pytest.mark.parametrize("cfg", [synth.TINY, SMALL_FP8], ids=["bf16", "fp8"])
def test_rejects_two_token_rows_swapped(cfg):
    c = _case(cfg)
    h = c["h_round"].copy()
    y = _y_from_h(c, h)
    y[[3, 11]] = y[[11, 3]]
    with pytest.raises(AssertionError, match="y elements"):
        _check(c, h, y)


def test_rejects_fp8_code_two_steps_off():
    c = _case(SMALL_FP8)
    orc = c["orc"]
    h = c["h_round"].copy()
    for n, j, i in _pick(h, 3 / h.size, 4):
        g0 = (i // 32) * 32
        e = orc.fp8_group_exponent(c["ref_h"][n, j, g0:g0 + 32])
        code = orc.e4m3_rne_sat(h[n, j, i] / 2.0 ** e)
        mag = min((code & 0x7F) + 2, 0x7E)
        h[n, j, i] = orc.e4m3_value((code & 0x80) | mag) * 2.0 ** e
    with pytest.raises(AssertionError, match="admissible"):
        _check(c, h, _y_from_h(c, h))
