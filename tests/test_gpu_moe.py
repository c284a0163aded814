"""GPU parity of prepare_weights (layout round trip) and moe_forward (S2-S7)
against the FP64 oracle, within |gpu - oracle| <= 2^-7|oracle| + 1e-3 rms."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import block_scaled_fp4_02_gb300 as fp4
import synth
from _util import (bf16_tensor, check_moe, decode_packed, decode_packed_mx,
                   dequant_reference,
                   requant_weights_oracle, weights_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    fp4.build()
    fp4.load()
    assert fp4.build_flags() == (fp4.BUILD_BOUNDS_CHECK
                                 if fp4.variant() == "checked" else 0)
    assert fp4.last_device_error() == fp4.OK


def to_dev(w):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda()
            for k, v in w.items()}


def prepare(w, gran=16, layout=0, act=fp4.ACT_BF16):
    d = to_dev(w)
    p = fp4.prepare_weights(d["w13"], d["w13_s"], d["w13_gs"], d["w2"],
                            d["w2_s"], d["w2_gs"], gran_k=gran,
                            w13_layout=layout, act_mode=act)
    del d
    return p


def swap_halves(w, I):
    out = dict(w)
    out["w13"] = np.ascontiguousarray(
        np.concatenate([w["w13"][:, I:], w["w13"][:, :I]], 1))
    out["w13_s"] = np.ascontiguousarray(
        np.concatenate([w["w13_s"][:, I:], w["w13_s"][:, :I]], 1))
    return out


def gpu_forward(p, acts, k, act):
    """moe_forward on device tensors; returns y and the workspace."""
    logits = torch.from_numpy(acts["logits"]).cuda()
    xb = bf16_tensor(acts["x_bf16"])
    T = logits.shape[0]
    ws = torch.empty(max(fp4.moe_workspace_size(p, T, k), 256),
                     dtype=torch.uint8, device="cuda")
    if act == fp4.ACT_BF16:
        y = fp4.moe_forward(xb, None, logits, p, k, workspace=ws)
    else:
        xq, xs = fp4.act_quant(xb)
        y = fp4.moe_forward(xq, xs, logits, p, k, workspace=ws)
    torch.cuda.synchronize()
    assert fp4.last_device_error() == fp4.OK
    return y, ws


def check_against_oracle(orc, cfg, w, acts, p, y, ws, tokens, layout=0,
                         gran=16, what=None, record=None):
    """Oracle rows for `tokens`, then the two-level (h, y) parity check."""
    tokens = list(tokens)
    if cfg.act == "fp8":
        w_used = requant_weights_oracle(orc, w, cfg.E, cfg.K, cfg.I)
        xq, xs = orc.act_quant(acts["x_bf16"])
        ref_y, ref_h, aux = orc.moe_rows(tokens, **w_used, gran=32,
                                    w13_layout=layout, act_mode=1,
                                    top_k=cfg.top_k, logits=acts["logits"],
                                    xq=xq, xs=xs, return_h=True)
        gran, act = 32, 1
    else:
        w_used, act = w, 0
        ref_y, ref_h, aux = orc.moe_rows(tokens, **w, gran=gran,
                                    w13_layout=layout, act_mode=0,
                                    top_k=cfg.top_k, logits=acts["logits"],
                                    x_bf16=acts["x_bf16"], return_h=True)
    return check_moe(orc, fp4, cfg, p, y, ws, tokens, ref_y, ref_h, aux,
                     w_used, gran, act, acts["logits"], what or cfg.name,
                     record=record)


# ------------------------------------------------------------------ layout

@pytest.mark.parametrize("gran,act", [(16, fp4.ACT_BF16), (16, fp4.ACT_FP8),
                                      (16, fp4.ACT_FP8 | fp4.FLAG_KEEP_GROUP16),
                                      (32, fp4.ACT_BF16)])
@pytest.mark.parametrize("layout", [0, 1])
def test_prepare_layout_roundtrip(orc, gran, act, layout):
    E, K, I = 3, 256, 384
    w = synth.moe_weights(synth.MoeConfig("rt", E, K, I, 1, 1, weight_seed=77))
    if gran == 32:
        w = requant_weights_oracle(orc, w, E, K, I)
    p = prepare(w, gran=gran, layout=layout, act=act)
    bufs = p.buffers()
    d = p.desc
    if act == fp4.ACT_FP8 and gran == 16:   # lossy requant to group32
        ref_w = requant_weights_oracle(orc, w, E, K, I)
        rg = 32
    else:
        ref_w, rg = w, gran
    assert d.gran_k == rg
    ref13 = dequant_reference(ref_w["w13"], ref_w["w13_s"], rg, ref_w["w13_gs"])
    ref2 = dequant_reference(ref_w["w2"], ref_w["w2_s"], rg, ref_w["w2_gs"])
    # FP8 activations over group32 weights: the block-scaled layout
    assert d.layout == (1 if (act & 0xFF) == fp4.ACT_FP8 and rg == 32 else 0)
    if d.layout == 1:
        got13 = decode_packed_mx(bufs["w13"].numpy(),
                                 bufs["w13_scales"].numpy(), E, 2 * I, K,
                                 bufs["alpha13"].numpy(), True, I, layout)
        got2 = decode_packed_mx(bufs["w2"].numpy(), bufs["w2_scales"].numpy(),
                                E, K, I, bufs["alpha2"].numpy(), False)
    else:
        got13 = decode_packed(bufs["w13"].numpy(), E, 2 * I, K, rg,
                              d.scale_mul, d.scale_add,
                              bufs["alpha13"].numpy(), True, I, layout)
        got2 = decode_packed(bufs["w2"].numpy(), E, K, I, rg, d.scale_mul,
                             d.scale_add, bufs["alpha2"].numpy(), False)
    # Exact: every packed value equals e2m1 * scale * gs of the source.
    np.testing.assert_array_equal(got13, ref13)
    np.testing.assert_array_equal(got2, ref2)


def test_prepare_rejects_nan_scale():
    E, K, I = 2, 128, 128
    w = synth.moe_weights(synth.MoeConfig("nan", E, K, I, 1, 1, weight_seed=5))
    w["w2_s"][1, 7, 3] = 0x7F
    with pytest.raises(fp4.FP4MoEError) as ei:
        prepare(w)
    assert ei.value.code == fp4.ERR_INVALID_ARG


# --------------------------------------------------------------- MoE small

SMALL = [synth.TINY, synth.SMALL_DECODE, synth.SMALL_PREFILL, synth.SMALL_FP8]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("layout", [0, 1])
def test_moe_small_configs_all_tokens(orc, cfg, layout, record_property):
    w = weights_for(cfg)
    if layout == 1:
        w = swap_halves(w, cfg.I)
    acts = synth.moe_activations(cfg)
    act = fp4.ACT_FP8 if cfg.act == "fp8" else fp4.ACT_BF16
    p = prepare(w, layout=layout, act=act)
    y, ws = gpu_forward(p, acts, cfg.top_k, act)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, range(cfg.T),
                         layout=layout,
                         record=record_property)


def test_moe_group32_weights_bf16_activations(orc, record_property):
    # W4A16 over MX (UE8M0 group32) weights, no requant on the GPU side.
    cfg = synth.SMALL_DECODE
    w32 = requant_weights_oracle(orc, weights_for(cfg), cfg.E, cfg.K, cfg.I)
    acts = synth.moe_activations(cfg)
    p = prepare(w32, gran=32)
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    check_against_oracle(orc, cfg, w32, acts, p, y, ws, range(cfg.T), gran=32,
                         what="group32 bf16",
                         record=record_property)


def _fp8_group16_oracle(orc, cfg, w, acts, tokens):
    xq, xs = orc.act_quant(acts["x_bf16"])
    return orc.moe_rows(tokens, **w, gran=16, w13_layout=0, act_mode=1,
                        top_k=cfg.top_k, logits=acts["logits"], xq=xq, xs=xs,
                        return_h=True)


def test_moe_fp8_keep_group16(orc, record_property):
    # FP8 activations over group16 weights without the lossy requant: the
    # oracle runs the group16 weights as they are.
    cfg = synth.SMALL_FP8
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w, act=fp4.ACT_FP8 | fp4.FLAG_KEEP_GROUP16)
    assert p.desc.gran_k == 16 and p.desc.act_mode == fp4.ACT_FP8
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_FP8)
    tokens = list(range(cfg.T))
    ref_y, ref_h, aux = _fp8_group16_oracle(orc, cfg, w, acts, tokens)
    check_moe(orc, fp4, cfg, p, y, ws, tokens, ref_y, ref_h, aux, w, 16, 1,
              acts["logits"], "fp8 keep group16", record=record_property)


def test_fp8_group16_accuracy_gap(orc, record_property):
    # Against the exact FP64 result over the group16 weights, the kept
    # group16 path errs only by its roundings; the requant path adds the
    # group32 re-rounding of the weights.  Relative RMS errors are recorded.
    cfg = synth.SMALL_FP8
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    tokens = list(range(cfg.T))
    ref_y = _fp8_group16_oracle(orc, cfg, w, acts, tokens)[0].reshape(cfg.T, cfg.K)
    errs = {}
    for name, mode in (("keep_group16", fp4.ACT_FP8 | fp4.FLAG_KEEP_GROUP16),
                       ("requant_group32", fp4.ACT_FP8)):
        p = prepare(w, act=mode)
        y, _ = gpu_forward(p, acts, cfg.top_k, fp4.ACT_FP8)
        d = y.float().cpu().numpy().astype(np.float64) - ref_y
        errs[name] = float(np.sqrt((d ** 2).mean() / (ref_y ** 2).mean()))
        record_property(name + "_rel_rms", errs[name])
        del p
    print("fp8 relative RMS error vs exact group16:", errs)
    assert errs["keep_group16"] < 2.0 ** -7
    assert errs["keep_group16"] < errs["requant_group32"]


def test_moe_inverted_global_scales():
    # Compressed-tensors checkpoints store 1/gs: with the flag, prepare takes
    # the reciprocal (FP32 division), so the layer equals the one prepared
    # from the reciprocal computed on the host, bit for bit.
    cfg = synth.SMALL_DECODE
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    inv = dict(w)
    for k in ("w13_gs", "w2_gs"):
        inv[k] = (np.float32(1.0) / w[k].astype(np.float32)).astype(np.float32)
    direct = dict(w)
    for k in ("w13_gs", "w2_gs"):
        direct[k] = (np.float32(1.0) / inv[k]).astype(np.float32)
    p_inv = prepare(inv, act=fp4.ACT_BF16 | fp4.FLAG_GS_INVERTED)
    p_dir = prepare(direct)
    y_inv, _ = gpu_forward(p_inv, acts, cfg.top_k, fp4.ACT_BF16)
    y_dir, _ = gpu_forward(p_dir, acts, cfg.top_k, fp4.ACT_BF16)
    assert torch.equal(y_inv.view(torch.int16), y_dir.view(torch.int16))
    a_inv = p_inv.buffers()["alpha13"].numpy()
    a_dir = p_dir.buffers()["alpha13"].numpy()
    np.testing.assert_array_equal(a_inv, a_dir)


@pytest.mark.parametrize("T", [1, 2, 17, 300])
def test_moe_token_counts(orc, T, record_property):
    base = synth.SMALL_DECODE
    cfg = synth.MoeConfig("t", base.E, base.K, base.I, T, base.top_k,
                          weight_seed=base.weight_seed, input_seed=900 + T)
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w)
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, range(T), what=f"T={T}",
                         record=record_property)


@pytest.mark.parametrize("k", [1, 2])
def test_moe_hot_experts_get_every_token(orc, k, record_property):
    # The first k experts win every token: 600 tokens per expert, so each
    # expert is split into several token chunks.
    cfg = synth.MoeConfig("hot", 8, 768, 384, 600, k, weight_seed=3002,
                          input_seed=4242)
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    acts["logits"][:, 0] += 100.0
    acts["logits"][:, 1] += 99.0
    p = prepare(w)
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, range(cfg.T),
                         what=f"hot experts k={k}",
                         record=record_property)


def test_moe_zero_tokens_is_noop():
    cfg = synth.TINY
    p = prepare(weights_for(cfg))
    x = torch.empty(0, cfg.K, dtype=torch.bfloat16, device="cuda")
    logits = torch.empty(0, cfg.E, dtype=torch.float32, device="cuda")
    y = fp4.moe_forward(x, None, logits, p, cfg.top_k,
                        workspace=torch.empty(256, dtype=torch.uint8,
                                              device="cuda"))
    assert y.shape == (0, cfg.K)


def test_moe_deterministic_and_host_api(orc):
    cfg = synth.SMALL_PREFILL
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w)
    y1, _ = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    y2, _ = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # the host-buffer entry point gives the same bits
    xh = torch.from_numpy(acts["x_bf16"].view(np.int16)).view(
        torch.bfloat16).pin_memory()
    lh = torch.from_numpy(acts["logits"]).pin_memory()
    yh = torch.empty(cfg.T, cfg.K, dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(fp4.moe_workspace_size_host(p, cfg.T, cfg.top_k),
                     dtype=torch.uint8, device="cuda")
    fp4.moe_forward_host(xh, None, lh, p, cfg.top_k, yh, ws)
    torch.cuda.synchronize()
    assert torch.equal(yh.view(torch.int16), y1.cpu().view(torch.int16))


@pytest.mark.parametrize("cfg", [synth.SMALL_DECODE, synth.SMALL_PREFILL, synth.SMALL_FP8],
                         ids=lambda c: c.name)
def test_moe_forward_graph_replay(cfg):
    """moe_forward makes no host synchronisation or allocation after its
    first call on a device, so it can be captured into a CUDA graph (how a
    serving loop removes the per-call launch cost at a few tokens).  A
    replay gives the eager call's bits, for the captured inputs and for new
    inputs copied into the same buffers."""
    w = weights_for(cfg)
    act = fp4.ACT_FP8 if cfg.act == "fp8" else fp4.ACT_BF16
    p = prepare(w, act=act)
    k = cfg.top_k

    def device_inputs(c):
        acts = synth.moe_activations(c)
        xb = bf16_tensor(acts["x_bf16"])
        if act == fp4.ACT_FP8:
            xq, xs = fp4.act_quant(xb)
            return xq, xs, torch.from_numpy(acts["logits"]).cuda()
        return xb, None, torch.from_numpy(acts["logits"]).cuda()

    ws_bytes = max(fp4.moe_workspace_size(p, cfg.T, k), 256)

    def eager(x, xs, lg):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        y = fp4.moe_forward(x, xs, lg, p, k, workspace=ws)
        torch.cuda.synchronize()
        return y

    x0, xs0, lg0 = device_inputs(cfg)
    other = dataclasses.replace(cfg, input_seed=cfg.input_seed + 17)
    x1, xs1, lg1 = device_inputs(other)
    y_ref0, y_ref1 = eager(x0, xs0, lg0), eager(x1, xs1, lg1)
    # static buffers of the graph
    xg, lgg = x0.clone(), lg0.clone()
    xsg = xs0.clone() if xs0 is not None else None
    yg = torch.empty_like(y_ref0)
    wsg = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):       # warm-up call on the capture stream
        fp4.moe_forward(xg, xsg, lgg, p, k, y=yg, workspace=wsg)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fp4.moe_forward(xg, xsg, lgg, p, k, y=yg, workspace=wsg)
    yg.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fp4.last_device_error() == fp4.OK
    assert torch.equal(yg.view(torch.int16), y_ref0.view(torch.int16))
    xg.copy_(x1)
    lgg.copy_(lg1)
    if xsg is not None:
        xsg.copy_(xs1)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yg.view(torch.int16), y_ref1.view(torch.int16))


@pytest.mark.parametrize("E,T,k,K,I,act", [
    (8, 16, 2, 256, 256, fp4.ACT_BF16), (32, 13, 4, 256, 256, fp4.ACT_BF16),
    (256, 1, 8, 256, 256, fp4.ACT_BF16), (256, 32, 8, 256, 256, fp4.ACT_BF16),
    (64, 32, 16, 256, 256, fp4.ACT_BF16), (1024, 7, 8, 128, 128, fp4.ACT_BF16),
    (32, 13, 4, 256, 256, fp4.ACT_FP8), (256, 32, 8, 256, 256, fp4.ACT_FP8)])
def test_moe_few_tokens_routing_matches_three_kernels(E, T, k, K, I, act):
    """Up to 32 tokens, moe_forward routes, scans and scatters in one launch;
    its ids, weights, counts, offsets, perm and inv equal route_debug's
    (route, scan and scatter as three kernels) bit for bit, with many tied
    logits."""
    cfg = synth.MoeConfig(f"few_tokens_E{E}_T{T}_k{k}", E, K, I, T, k,
                          weight_seed=3201, input_seed=3301 + T)
    p = prepare(weights_for(cfg), act=act)
    acts = synth.moe_activations(cfg)
    logits = (np.round(acts["logits"] * 4) / 4).astype(np.float32)
    lg = torch.from_numpy(logits).cuda()
    xb = bf16_tensor(acts["x_bf16"])
    ws = torch.empty(max(fp4.moe_workspace_size(p, T, k), 256), dtype=torch.uint8,
                     device="cuda")
    if act == fp4.ACT_BF16:
        fp4.moe_forward(xb, None, lg, p, k, workspace=ws)
    else:
        xq, xs = fp4.act_quant(xb)
        fp4.moe_forward(xq, xs, lg, p, k, workspace=ws)
    torch.cuda.synchronize()
    assert fp4.last_device_error() == fp4.OK
    ref = fp4.route_debug(lg, k)
    offs = fp4.moe_workspace_offsets(p, T, k)
    P = T * k

    def region(name, n):
        return ws[offs[name]:offs[name] + 4 * n].view(torch.int32)

    assert torch.equal(region("ids", P), ref["ids"].view(-1))
    assert torch.equal(region("w", P), ref["w"].view(-1).view(torch.int32))
    assert torch.equal(region("counts", E), ref["counts"])
    assert torch.equal(region("offsets", E + 1), ref["offsets"])
    assert torch.equal(region("perm", P), ref["perm"])
    assert torch.equal(region("inv", P), ref["inv"])


def test_moe_host_api_two_streams():
    """Calls on two streams at once, each with its own workspace and output
    buffer (how the end-to-end measurement overlaps one step's copies with
    the other's kernels), give the one-stream bits: the forward keeps no
    device state between calls but the status word."""
    cfg = synth.SMALL_PREFILL
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w)
    y_ref, _ = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    other = dataclasses.replace(cfg, input_seed=cfg.input_seed + 5)
    acts2 = synth.moe_activations(other)
    y_ref2, _ = gpu_forward(p, acts2, cfg.top_k, fp4.ACT_BF16)

    def host(a):
        xh = torch.from_numpy(a["x_bf16"].view(np.int16)).view(torch.bfloat16).pin_memory()
        return xh, torch.from_numpy(a["logits"]).pin_memory()

    ins = [host(acts), host(acts2)]
    refs = [y_ref.cpu(), y_ref2.cpu()]
    n = fp4.moe_workspace_size_host(p, cfg.T, cfg.top_k)
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [[torch.empty(cfg.T, cfg.K, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
            for _ in range(2)]
    for i in range(3):
        for j in range(2):
            fp4.moe_forward_host(ins[j][0], None, ins[j][1], p, cfg.top_k, outs[j][i],
                                 wss[j], stream=streams[j])
    torch.cuda.synchronize()
    assert fp4.last_device_error() == fp4.OK
    for j in range(2):
        for i in range(3):
            assert torch.equal(outs[j][i].view(torch.int16), refs[j].view(torch.int16))


def test_moe_workspace_too_small():
    cfg = synth.TINY
    p = prepare(weights_for(cfg))
    acts = synth.moe_activations(cfg)
    need = fp4.moe_workspace_size(p, cfg.T, cfg.top_k)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp4.FP4MoEError) as ei:
        fp4.moe_forward(bf16_tensor(acts["x_bf16"]), None,
                        torch.from_numpy(acts["logits"]).cuda(), p,
                        cfg.top_k, workspace=ws)
    assert ei.value.code == fp4.ERR_WORKSPACE_TOO_SMALL


# ---------------------------------------------------------- MoE full size

def _sample_tokens(T, n, seed):
    g = np.random.default_rng(seed)
    s = set(g.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return sorted(s)


# Few-token decode at full size (8 and ~32 experts touched), same weights as
# the decode workload.
DECODE_T1 = synth.MoeConfig("decode_w4a16_E256_K6144_I2048_T1_k8", 256, 6144, 2048, 1, 8,
                            weight_seed=1003, input_seed=2021)
DECODE_T4 = synth.MoeConfig("decode_w4a16_E256_K6144_I2048_T4_k8", 256, 6144, 2048, 4, 8,
                            weight_seed=1003, input_seed=2022)


@pytest.mark.parametrize("cfg,n", [(synth.DECODE, 64), (synth.DECODE_SKEW, 64),
                                   (DECODE_T1, 1), (DECODE_T4, 4),
                                   (synth.PREFILL, 24), (synth.FP8, 24)],
                         ids=lambda c: getattr(c, "name", str(c)))
def test_moe_full_size_sampled(orc, cfg, n, record_property):
    """Full-size workloads in the benchmark's launch configuration; the
    oracle recomputes a sample of output rows one token at a time."""
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    act = fp4.ACT_FP8 if cfg.act == "fp8" else fp4.ACT_BF16
    p = prepare(w, act=act)
    y, ws = gpu_forward(p, acts, cfg.top_k, act)
    toks = _sample_tokens(cfg.T, n, 99)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, toks,
                         record=record_property)
    p.free()


def test_moe_full_size_fp8_keep_group16(orc, record_property):
    """The FP8 workload with its group16 weights kept (no requant), sampled
    rows against the oracle over the group16 weights."""
    cfg = synth.FP8
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w, act=fp4.ACT_FP8 | fp4.FLAG_KEEP_GROUP16)
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_FP8)
    toks = _sample_tokens(cfg.T, 24, 98)
    ref_y, ref_h, aux = _fp8_group16_oracle(orc, cfg, w, acts, toks)
    check_moe(orc, fp4, cfg, p, y, ws, toks, ref_y, ref_h, aux, w, 16, 1,
              acts["logits"], "fp8 keep group16, full size",
              record=record_property)
    p.free()


@pytest.mark.parametrize("E,K,I,T,k", [
    (1, 128, 128, 40, 1),     # smallest shapes: one K step pair, one expert
    (16, 256, 128, 50, 16),   # top_k = E = 16 (every expert, largest k)
    (3, 384, 256, 700, 3),    # many tokens, odd expert count, k = E
    (5, 128, 384, 90, 2),     # T in (64, 256]: 256-token chunks, few per expert
])
def test_moe_edge_shapes(orc, E, K, I, T, k, record_property):
    cfg = synth.MoeConfig(f"edge_E{E}_K{K}_I{I}_T{T}_k{k}", E, K, I, T, k,
                          weight_seed=5000 + E + K + I, input_seed=6000 + T)
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w)
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_BF16)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, range(T), what=cfg.name,
                         record=record_property)


@pytest.mark.parametrize("E,K,I,T,k", [
    (4, 384, 384, 100, 2),    # FC1 and FC2 on the one-CTA block-scaled kernel
    (3, 768, 256, 300, 3),    # FC1 on CTA pairs, FC2 (6 row blocks) on one CTA
])
def test_moe_fp8_edge_shapes(orc, E, K, I, T, k, record_property):
    # Block counts that do not split over CTA pairs take the one-CTA
    # block-scaled kernel.
    cfg = synth.MoeConfig(f"fp8_edge_E{E}_K{K}_I{I}_T{T}_k{k}", E, K, I, T, k,
                          act="fp8", weight_seed=5100 + E + K + I,
                          input_seed=6100 + T)
    w = weights_for(cfg)
    acts = synth.moe_activations(cfg)
    p = prepare(w, act=fp4.ACT_FP8)
    assert p.desc.layout == 1
    y, ws = gpu_forward(p, acts, cfg.top_k, fp4.ACT_FP8)
    check_against_oracle(orc, cfg, w, acts, p, y, ws, range(T), what=cfg.name,
                         record=record_property)
