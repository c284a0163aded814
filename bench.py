#!/usr/bin/env python3
"""Benchmark of the block-scaled FP4 MoE layer on GB300 (one JSON line).

A step is one pass of the hot path over one batch of synthetic input:
routing, permutation + gather, FC1 gate|up + SwiGLU, FC2 and the weighted
combine (plus the FP8 activation quantization and the FP8 rounding of the
intermediate in the FP8 workload), all through the C ABI.  The headline
workload is the prefill-shaped W4A16 layer (E256 K6144 I2048 top-8,
T = 8192 tokens); the decode, skewed-decode, FP8 x FP4 and requant workloads
are reported under "extra".  Inputs stay resident in HBM; the packed
weights (5.4 GB) exceed L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs an independent replica (the layer does not
shard across GPUs here); the value is all ranks' tokens over the slowest
rank's time.  `--impl reference` times the FP64 CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("MoE-layer tokens/s, TFLOP/s & weight GB/s vs GB300 roofline; "
          "requant GB/s")
WORKLOADS = {"prefill": synth.PREFILL, "decode": synth.DECODE,
             "decode_skew": synth.DECODE_SKEW, "fp8": synth.FP8,
             # FP8 activations over the group16 weights without the requant
             "fp8_g16": synth.MoeConfig(
                 "fp8xfp4_group16_E128_K7168_I2048_T4096_k8", 128, 7168, 2048,
                 4096, 8, act="fp8", weight_seed=1005, input_seed=2005,
                 keep_group16=True),
             "tiny": synth.TINY,
             # small-M decode on the decode weights (T = 1, 4, 16 tokens)
             "decode_t1": synth.MoeConfig(
                 "decode_w4a16_E256_K6144_I2048_T1_k8", 256, 6144, 2048, 1, 8,
                 weight_seed=1003, input_seed=2101),
             "decode_t4": synth.MoeConfig(
                 "decode_w4a16_E256_K6144_I2048_T4_k8", 256, 6144, 2048, 4, 8,
                 weight_seed=1003, input_seed=2104),
             "decode_t16": synth.MoeConfig(
                 "decode_w4a16_E256_K6144_I2048_T16_k8", 256, 6144, 2048, 16,
                 8, weight_seed=1003, input_seed=2116),
             # small cases of the same kernels for ncu captures: inputs larger
             # than L2, a few GB on the device at most, and 19 experts so
             # the GEMM work units are a multiple of the 152 SMs (no tail)
             "prefill_small": synth.MoeConfig(
                 "prefill_small_w4a16_E19_K6144_I2048_T608_k8", 19, 6144, 2048,
                 608, 8, weight_seed=1013, input_seed=2024),
             "decode_small": synth.MoeConfig(
                 "decode_small_w4a16_E19_K6144_I2048_T8_k8", 19, 6144, 2048, 8,
                 8, weight_seed=1023, input_seed=2035),
             "fp8_small": synth.MoeConfig(
                 "fp8_small_E19_K7168_I2048_T608_k8", 19, 7168, 2048, 608, 8,
                 act="fp8", weight_seed=1015, input_seed=2025)}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fp4moe",
                    choices=["fp4moe", "reference"])
    ap.add_argument("--workload", default="prefill", choices=sorted(WORKLOADS))
    ap.add_argument("--extra", default="decode,decode_skew,decode_t1,decode_t4,"
                    "decode_t16,fp8,fp8_g16,requant",
                    help="comma list of extra workloads, or 'none'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev)], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 3.0:
            self.file.flush()
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.02)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 8:
                    rows.append(p)
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        sm, smax, reasons = [], [], set()
        for p in rows:
            try:
                sm.append(float(p[0]))
                smax.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------- GPU

class MoeRun:
    """One MoE workload resident on the GPU."""

    def __init__(self, cfg, fp4, torch, weights):
        self.cfg, self.fp4, self.torch = cfg, fp4, torch
        self.fp8 = cfg.act == "fp8"
        act = fp4.ACT_FP8 if self.fp8 else fp4.ACT_BF16
        if cfg.keep_group16:
            act |= fp4.FLAG_KEEP_GROUP16
        dev = {k: torch.from_numpy(v).cuda() for k, v in weights.items()}
        self.packed = fp4.prepare_weights(
            dev["w13"], dev["w13_s"], dev["w13_gs"], dev["w2"], dev["w2_s"],
            dev["w2_gs"], gran_k=16, w13_layout=cfg.w13_layout, act_mode=act)
        del dev
        acts = synth.moe_activations(cfg)
        self.acts = acts
        self.logits = torch.from_numpy(acts["logits"]).cuda()
        self.x = torch.from_numpy(acts["x_bf16"].view(np.int16)).cuda().view(
            torch.bfloat16)
        T = cfg.T
        self.y = torch.empty(T, cfg.K, dtype=torch.bfloat16, device="cuda")
        n = fp4.moe_workspace_size(self.packed, T, cfg.top_k)
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        if self.fp8:
            self.xq = torch.empty(T, cfg.K, dtype=torch.uint8, device="cuda")
            self.xs = torch.empty(T, cfg.K // 32, dtype=torch.uint8,
                                  device="cuda")
        r = fp4.route_debug(self.logits, cfg.top_k)
        self.touched = int((r["counts"] > 0).sum().item())
        torch.cuda.synchronize()
        d = self.packed.desc
        self.mx = d.layout == 1          # block-scaled path (FP8 x group32)
        self.w13_bytes_per_expert = (d.w13_bytes + d.w13_scales_bytes) // cfg.E
        self.w2_bytes_per_expert = (d.w2_bytes + d.w2_scales_bytes) // cfg.E

    def step(self):
        fp4 = self.fp4
        if self.fp8:
            fp4.act_quant(self.x, self.xq, self.xs)
            fp4.moe_forward(self.xq, self.xs, self.logits, self.packed,
                            self.cfg.top_k, self.y, self.ws)
        else:
            fp4.moe_forward(self.x, None, self.logits, self.packed,
                            self.cfg.top_k, self.y, self.ws)

    @property
    def launches_per_step(self) -> int:
        # act_quant, route, scan, scatter, gather, FC1, FC2, combine (FP8: the
        # block-scaled path rounds h inside FC1; kept group16 weights add the
        # separate rounding kernel)
        if self.fp8:
            return 9 if self.cfg.keep_group16 else 8
        return 7

    def timed(self, steps, warmup, clocks=None):
        """K steps with an event between stages (the per-stage times and,
        for steps of 2 ms or more, the step's value).  An event record
        between two kernels costs the stream ~2-3 us, so a shorter step is
        timed again as a whole, without them, for its value."""
        torch, fp4 = self.torch, self.fp4
        host = []
        for _ in range(warmup):
            th = time.perf_counter()
            self.step()
            host.append(time.perf_counter() - th)
        # the host's enqueue time of a step, first (module loading) call aside
        host_step = float(np.median(host[1:] if len(host) > 1 else host or [0.0]))
        torch.cuda.synchronize()
        ev = torch.cuda.Event
        stage = [[ev(enable_timing=True) for _ in range(fp4.STAGE_EVENTS)]
                 for _ in range(steps)]
        for row in stage:      # creates the underlying CUDA events
            for e in row:
                e.record()
        t0, t1 = ev(enable_timing=True), ev(enable_timing=True)
        torch.cuda.synchronize()

        # A small step's launches can take the host longer to enqueue than
        # the device to run (T <= 16 tokens): the timed steps queue behind a
        # device-side delay that outlasts their enqueueing (with stage events
        # a step takes the host longer than in the warm-up: a factor of 3),
        # so the events measure device time.
        def delay():
            torch.cuda._sleep(int((3.0 * steps * host_step + 2e-3) * 2.2e9))

        def run(with_stages):
            delay()
            t0.record()
            for i in range(steps):
                if with_stages:
                    fp4.set_stage_events(stage[i])
                self.step()
            t1.record()
            torch.cuda.synchronize()
            assert fp4.last_device_error() == fp4.OK
            return t0.elapsed_time(t1)

        if clocks:
            clocks.start()
        total_ms = run(True)
        if total_ms / steps < 2.0:
            total_ms = run(False)
        clk = clocks.stop() if clocks else None
        per_stage = np.zeros(fp4.STAGE_EVENTS - 1)
        for row in stage:
            for j in range(fp4.STAGE_EVENTS - 1):
                per_stage[j] += row[j].elapsed_time(row[j + 1])
        per_stage /= steps
        return total_ms, dict(zip(fp4.STAGE_NAMES, per_stage.tolist())), clk

    def graph_timed(self, steps, warmup):
        """Device ms per step of a CUDA-graph replay of one step: how a
        serving loop runs a few tokens without the per-launch cost of eager
        calls (the forward makes no host synchronisation or allocation, so
        it captures as is)."""
        torch, fp4 = self.torch, self.fp4
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        host = []
        for _ in range(max(warmup, 1)):
            th = time.perf_counter()
            g.replay()
            host.append(time.perf_counter() - th)
        host_step = float(np.median(host))
        torch.cuda.synchronize()
        t0, t1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        torch.cuda._sleep(int((1.5 * steps * host_step + 5e-4) * 2.2e9))
        t0.record()
        for _ in range(steps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        assert fp4.last_device_error() == fp4.OK
        del g
        return t0.elapsed_time(t1) / steps

    def e2e(self, steps, warmup):
        """Steps through the host-buffer entry point: each step copies its
        inputs from pinned host memory, runs the layer and copies y back.
        Two streams, each with its own workspace and output buffer, take
        the steps in turn, so that one step's copies overlap the other's
        kernels (the copy engines and the SMs work at once)."""
        torch, fp4, cfg = self.torch, self.fp4, self.cfg
        if self.fp8:
            fp4.act_quant(self.x, self.xq, self.xs)
            xh = self.xq.cpu().pin_memory()
            sh = self.xs.cpu().pin_memory()
        else:
            xh = self.x.cpu().pin_memory()
            sh = None
        lh = self.logits.cpu().pin_memory()
        nws = fp4.moe_workspace_size_host(self.packed, cfg.T, cfg.top_k)
        streams = [torch.cuda.Stream() for _ in range(2)]
        yhs = [torch.empty(cfg.T, cfg.K, dtype=torch.bfloat16).pin_memory()
               for _ in range(2)]
        wss = [torch.empty(nws, dtype=torch.uint8, device="cuda")
               for _ in range(2)]

        def one(i):
            fp4.moe_forward_host(xh, sh, lh, self.packed, cfg.top_k,
                                 yhs[i % 2], wss[i % 2], stream=streams[i % 2])

        for i in range(warmup):
            one(i)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        t0.record(cur)
        for s in streams:
            s.wait_event(t0)
        for i in range(steps):
            one(i)
        for s in streams:
            cur.wait_stream(s)
        t1.record(cur)
        torch.cuda.synchronize()
        assert fp4.last_device_error() == fp4.OK
        ms = t0.elapsed_time(t1)
        h2d = xh.numel() * xh.element_size() + lh.numel() * 4 + (
            sh.numel() if sh is not None else 0)
        d2h = yhs[0].numel() * 2
        del wss
        return ms, h2d, d2h

    def weight_bytes(self) -> int:
        return self.touched * (self.w13_bytes_per_expert +
                               self.w2_bytes_per_expert)

    def _act_bytes(self, n: int) -> float:
        """Bytes of one gathered activation (or h) row of n elements: bf16,
        FP32 h on the kept-group16 FP8 path, E4M3 + one UE8M0 byte per 32 on
        the block-scaled path."""
        return n * (1 + 1 / 32) if self.mx else n * 2

    def fc1_bytes(self) -> int:
        """Algorithmic FC1 bytes: touched experts' packed FC1 weights, the
        gathered activations read once and h written once."""
        c = self.cfg
        P = c.T * c.top_k
        h = P * c.I * 4 if (self.fp8 and not self.mx) else P * self._act_bytes(c.I)
        return int(self.touched * self.w13_bytes_per_expert +
                   P * self._act_bytes(c.K) + h)

    def fc2_bytes(self) -> int:
        """Algorithmic FC2 bytes: touched experts' packed FC2 weights, h read
        once and the FP32 FC2 output written once."""
        c = self.cfg
        P = c.T * c.top_k
        return int(self.touched * self.w2_bytes_per_expert +
                   P * self._act_bytes(c.I) + P * c.K * 4)

    def free(self):
        self.packed.free()


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_moe_gemm_fc1.json")


def measured_traffic(workload: str):
    """FC1 DRAM bytes per launch from the committed ncu capture (scaled
    from a small case, see the file), or None when the sources of that
    workload's FC1 kernel have changed since the capture or no capture
    covers this workload."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        entry = t["per_launch_bytes"].get(workload)
        if entry is None:
            return None
        h = hashlib.sha256()
        for rel in entry["source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != entry["source_sha256"]:
            return None
        return float(entry["bytes"])
    except (OSError, KeyError, ValueError):
        return None


def tensor_peak(pk, fp8: bool):
    """Dense tensor peak for the workload's arithmetic: the measured bf16
    burst (a step of a few ms is timed, not a seconds-long loop); for the
    FP8 x FP4 workload, whose roofline is the FP8 dense rate, twice that (the
    nominal FP8 : bf16 ratio, 4.5 : 2.25 PFLOP/s)."""
    bf16 = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return (2.0 * bf16 if fp8 else bf16), bf16


def summarize(run: MoeRun, total_ms, stages, steps, pk, pk_src):
    cfg = run.cfg
    s = total_ms / 1e3
    tok = cfg.T * steps / s
    tflops = cfg.flops * steps / s / 1e12
    wgbs = run.weight_bytes() * steps / s / 1e9
    fc1_ms, fc2_ms = stages["fc1_swiglu"], stages["fc2"]
    P = cfg.T * cfg.top_k
    fc1_flops = 4 * cfg.K * cfg.I * P
    fc2_flops = 2 * cfg.K * cfg.I * P
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out = {"tokens_per_s": tok, "ms_per_step": total_ms / steps,
           "tflops": tflops, "weight_gbs": wgbs,
           "touched_experts": run.touched, "stage_ms": stages}
    tensor_bound = P / cfg.E >= 64
    # The FC1 kernel this workload runs: the block-scaled CTA-pair kernel for
    # FP8 activations over group32 weights, else the bf16 CTA-pair kernel for
    # chunks of up to 256 tokens (T > 64), else the one-CTA 32-token variant.
    if run.mx:
        kname = "moe_gemm_mx_pair_kernel<FC1> (FC1 + SwiGLU, block-scaled FP8 x FP4, CTA pairs)"
    elif cfg.T > 64:
        kname = "moe_gemm_pair_kernel<FC1> (FC1 + SwiGLU, CTA pairs)"
    else:
        kname = "moe_gemm_kernel<32, FC1> (FC1 + SwiGLU)"
    peak, bf16 = tensor_peak(pk, run.fp8)
    pname = ("2 x measured bf16_tflops (FP8 dense)" if run.fp8 else
             "bf16_tflops (burst)")
    if tensor_bound:
        ach = fc1_flops / (fc1_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": f"{pk_src} {pname}",
                "kernel": kname,
                "per_launch_flops": fc1_flops,
                "per_launch_bytes": run.fc1_bytes()}
        fc2 = fc2_flops / (fc2_ms / 1e3) / 1e12
        out["fc2_roofline"] = {"bound": "tensor", "achieved": fc2,
                               "peak": peak, "unit": "TFLOP/s",
                               "frac": fc2 / peak}
        out["layer_tensor_frac"] = tflops / peak
        if run.fp8:
            out["frac_vs_bf16_peak"] = {"fc1": ach / bf16, "fc2": fc2 / bf16,
                                        "layer": tflops / bf16}
    else:
        ach = run.fc1_bytes() / (fc1_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": f"{pk_src} hbm_gbs",
                "kernel": kname,
                "per_launch_bytes": run.fc1_bytes()}
        fc2 = run.fc2_bytes() / (fc2_ms / 1e3) / 1e9
        out["fc2_roofline"] = {"bound": "hbm", "achieved": fc2, "peak": hbm,
                               "unit": "GB/s", "frac": fc2 / hbm,
                               "per_launch_bytes": run.fc2_bytes()}
    roof["traffic"] = measured_traffic(cfg.name)
    out["layer_hbm_frac"] = wgbs / hbm
    return out, roof


def run_requant(fp4, torch, steps, warmup, pk):
    cfg = synth.REQUANT
    codes, scales, _ = synth.requant_inputs(cfg)
    c = torch.from_numpy(codes).cuda()
    s = torch.from_numpy(scales).cuda()
    oc = torch.empty_like(c)
    osc = torch.empty(cfg.rows, cfg.K // 32, dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        fp4.requant_fp4_gran_k(c, s, oc, osc)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        fp4.requant_fp4_gran_k(c, s, oc, osc)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    gbs = cfg.bytes_moved / (ms / 1e3) / 1e9
    peak = float(pk.get("hbm_gbs", 6800.0))
    return {"workload": cfg.name, "gbs": gbs, "ms_per_call": ms,
            "hbm_frac": gbs / peak, "bytes_per_call": cfg.bytes_moved}


# ------------------------------------------------------------------- CPU

def oracle_moe_sample(cfg, weights, seconds=12.0, max_tokens=256):
    """Times the FP64 oracle on a bounded number of tokens of the workload."""
    import oracle
    acts = synth.moe_activations(cfg)
    kw = dict(gran=16, w13_layout=cfg.w13_layout, act_mode=0, top_k=cfg.top_k,
              logits=acts["logits"], x_bf16=acts["x_bf16"])
    w = weights
    if cfg.act == "fp8":
        E, K, I = cfg.E, cfg.K, cfg.I
        c13, s13 = oracle.requant(w["w13"].reshape(-1, K // 2),
                                  w["w13_s"].reshape(-1, K // 16))
        c2, s2 = oracle.requant(w["w2"].reshape(-1, I // 2),
                                w["w2_s"].reshape(-1, I // 16))
        w = dict(w13=c13.reshape(E, 2 * I, K // 2),
                 w13_s=s13.reshape(E, 2 * I, K // 32), w13_gs=w["w13_gs"],
                 w2=c2.reshape(E, K, I // 2), w2_s=s2.reshape(E, K, I // 32),
                 w2_gs=w["w2_gs"])
        xq, xs = oracle.act_quant(acts["x_bf16"])
        kw.update(gran=32, act_mode=1, x_bf16=None, xq=xq, xs=xs)
    t = time.perf_counter()
    oracle.moe_rows([0], **w, **kw)
    per_tok = time.perf_counter() - t
    n = int(max(1, min(max_tokens, cfg.T, seconds / max(per_tok, 1e-6))))
    toks = list(range(n))
    t = time.perf_counter()
    oracle.moe_rows(toks, **w, **kw)
    dt = time.perf_counter() - t
    return {"value": n / dt, "unit": "tokens/s", "cores": oracle.cores(),
            "kind": "oracle",
            "sample": f"{n} of {cfg.T} tokens of {cfg.name}, FP64, "
                      f"{dt:.1f} s"}


def reference_arm(args):
    """--impl reference: the FP64 oracle on host cores, bounded samples."""
    import oracle
    oracle.build()
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = WORKLOADS[args.workload]
    weights = synth.moe_weights(cfg)
    budget = 120.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_moe_sample(cfg, weights, seconds=min(budget, 5.0),
                          max_tokens=4)
    vals, samples = [], []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        r = oracle_moe_sample(cfg, weights, seconds=budget, max_tokens=64)
        vals.append(r["value"])
        samples.append(r["sample"])
    wall = time.perf_counter() - t_all
    v = float(statistics.median(vals))
    line = {"impl": "reference", "metric": METRIC, "value": v,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": cfg.name, "T": cfg.T, "E": cfg.E,
                       "K": cfg.K, "I": cfg.I, "top_k": cfg.top_k,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": v, "unit": "tokens/s",
                             "cores": oracle.cores(), "kind": "oracle",
                             "sample": samples[-1] if samples else ""},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main

def main():
    args = parse_args()
    if args.impl == "reference":
        reference_arm(args)
        return
    import torch
    import block_scaled_fp4_02_gb300 as fp4

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    fp4.build()
    fp4.load()
    fp4.last_device_error()
    pk, pk_src = peaks()

    cfg = WORKLOADS[args.workload]
    weights = synth.moe_weights(cfg)
    run = MoeRun(cfg, fp4, torch, weights)
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms, stages, clk = run.timed(args.steps, args.warmup, clocks)
    if dist:
        t = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    head, roof = summarize(run, total_ms, stages, args.steps, pk, pk_src)

    e2e = None
    if not args.no_e2e:
        ms, h2d, d2h = run.e2e(args.steps, args.warmup)
        if dist:
            t = torch.tensor([ms], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        e2e = {"value": cfg.T * args.steps * world / (ms / 1e3),
               "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps,
               "streams": 2}

    extra = {}
    names = [] if args.extra == "none" else [
        n for n in args.extra.split(",") if n and n != args.workload]
    shared = {(cfg.E, cfg.K, cfg.I, cfg.weight_seed): run}
    for name in names:
        if name == "requant":
            extra["requant"] = run_requant(fp4, torch, args.steps,
                                           args.warmup, pk)
            continue
        c = WORKLOADS[name]
        key = (c.E, c.K, c.I, c.weight_seed)
        if (key in shared and shared[key].cfg.act == c.act and
                shared[key].cfg.keep_group16 == c.keep_group16):
            # same weights: reuse the packed set, new activations/routing
            base = shared[key]
            r = MoeRun.__new__(MoeRun)
            r.__dict__.update(base.__dict__)
            r.cfg = c
            acts = synth.moe_activations(c)
            r.logits = torch.from_numpy(acts["logits"]).cuda()
            r.x = torch.from_numpy(acts["x_bf16"].view(np.int16)).cuda().view(
                torch.bfloat16)
            r.y = torch.empty(c.T, c.K, dtype=torch.bfloat16, device="cuda")
            r.ws = torch.empty(fp4.moe_workspace_size(r.packed, c.T, c.top_k),
                               dtype=torch.uint8, device="cuda")
            rr = fp4.route_debug(r.logits, c.top_k)
            r.touched = int((rr["counts"] > 0).sum().item())
        else:
            r = MoeRun(c, fp4, torch, synth.moe_weights(c))
        ms, st, _ = r.timed(args.steps, args.warmup)
        sm, rf = summarize(r, ms, st, args.steps, pk, pk_src)
        sm["roofline"] = rf
        sm["workload"] = c.name
        if c.T <= 64:
            gms = r.graph_timed(args.steps, args.warmup)
            sm["graph_replay"] = {"ms_per_step": gms, "tokens_per_s": c.T / gms * 1e3,
                                  "layer_hbm_frac": r.weight_bytes() / (gms / 1e3) / 1e9
                                  / float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))}
        extra[name] = sm
        if r.packed is not run.packed:
            r.free()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cpu = oracle_moe_sample(cfg, weights)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": head["tokens_per_s"] * world,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, "
        "N(0,0.02) weights encoded NVFP4 group16)",
        "config": {"workload": cfg.name, "T": cfg.T, "E": cfg.E, "K": cfg.K,
                   "I": cfg.I, "top_k": cfg.top_k, "weights": "NVFP4 g16",
                   "activations": cfg.act, "parallelism": "replicas",
                   "l2": "inputs larger than L2 (packed weights "
                         f"{(run.packed.desc.w13_bytes + run.packed.desc.w2_bytes) / 1e9:.2f} GB)",
                   "timing": "CUDA events on the launching stream, steps queued behind a "
                             "device-side delay; stage times from events between the stages "
                             "(a step under 2 ms valued by a second pass without them)"},
        "tflops": head["tflops"] * world, "weight_gbs": head["weight_gbs"],
        "layer_hbm_frac": head["layer_hbm_frac"],
        "layer_tensor_frac": head.get("layer_tensor_frac"),
        "fc2_roofline": head["fc2_roofline"],
        "stage_ms": head["stage_ms"], "touched_experts": run.touched,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": run.launches_per_step * args.steps,
        "clocks": clk, "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
