"""Benchmark: exact attention forward + backward on GB300.

One step = one pass of the whole hot path over one batch: attn_fwd_train
(O in bf16 and fp32, lse), attn_bwd_preprocess_o32 (D = rowsum(dO o O)) and
attn_bwd (main kernel + dQ convert) on the causal
B=2 H=16 N=8192 d=128 workload (Q, K scaled by 3 for peaked softmax rows),
bf16 inputs resident in HBM.  FLOPs per step follow the stated convention:
forward 4*B*H*N^2*d, forward+backward 10*B*H*N^2*d, each halved for causal.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The "e2e" entry is the same step through the public torch API with the data
on the host: every step uploads Q, K, V, dO from pinned host memory and
downloads O, lse, dQ, dK, dV, pipelined over two buffer sets with the copies
on their own streams (the next step's upload and the previous step's
download overlap the current step's kernels).

Prints ONE JSON line on rank 0.  The reference arm (--impl reference) times
the fp64 CPU oracle, as it stands, on the host cores over a bounded sample
of the same workload (256 query rows and 256 key columns of one head per
step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from io_aware_exact_gb300.inputs import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "attention TFLOPS fwd and fwd+bwd on 1 GB300, % of dense BF16 tensor peak"
L2_BYTES = 126 * 1024 * 1024


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_tflops": d.get("bf16_tflops"), "bf16_tflops_sustained":
                d.get("bf16_tflops_sustained"), "hbm_gbs": d.get("hbm_gbs"), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_max(value: float, device="cpu") -> float:
    """Maximum of `value` over all ranks (the value itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, max_ms: float) -> float:
    """Units per second of the whole job: every rank processes `units_per_rank`
    (weak scaling); the job takes as long as its slowest rank."""
    return world * units_per_rank / (max_ms * 1e-3)


def _timed_steps(stream, flush, fn, steps, warmup, nev):
    """Run fn(None) `warmup` times, then `steps` times with an L2 flush before
    each (outside the events) and nev CUDA events handed to fn; returns the
    events.  The flush kernel itself runs once before the timed loop, so its
    first launch is not inside the timed region."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn(None)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        fn(evs[i])
    torch.cuda.synchronize()
    return evs


class _Problem:
    """Device buffers of one dense workload and the calls of its steps."""

    def __init__(self, w, dev, rank=0, Hkv=None):
        import torch
        import io_aware_exact_gb300 as attn
        self.attn = attn
        self.w = w
        B, H, N, d = w.B, w.H, w.N, w.d
        self.Hkv = Hkv or H
        self.x = make_inputs(B, H, N, d, w.seed + 100 * rank, w.qk_mult, with_grad=True)
        for n in ("k", "v"):          # grouped K / V heads: keep the first Hkv of each batch entry
            self.x[n] = self.x[n][:, :self.Hkv].contiguous()
        self.q, self.k, self.v, self.dO = (self.x[n].to(dev) for n in ("q", "k", "v", "dO"))
        self.o = torch.empty_like(self.q)
        self.o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.D = torch.empty_like(self.lse)
        self.acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q), torch.empty_like(self.k),
                                     torch.empty_like(self.v))
        self.splits = (int(attn.lib().attn_gqa_split_hint(B, H, self.Hkv, N, int(w.causal)))
                       if self.Hkv != H else 1)
        self.part = (torch.empty((2, self.splits, B, self.Hkv, N, d), dtype=torch.float32,
                                 device=dev) if self.splits > 1 else None)

    def _args(self):
        w = self.w
        return w.B, w.H, w.N, w.d, w.causal, w.scale

    def fwd(self, s):
        P = lambda t: t.data_ptr()
        B, H, N, d, causal, scale = self._args()
        self.attn.attn_fwd(P(self.q), P(self.k), P(self.v), P(self.o), P(self.lse), B, H, N, d,
                           causal, scale, s, Hkv=self.Hkv)

    def bwd_main(self, s):
        P = lambda t: t.data_ptr()
        B, H, N, d, causal, scale = self._args()
        if self.splits > 1:
            self.attn._check(self.attn.lib().attn_bwd_gqa_split(
                P(self.q), P(self.k), P(self.v), P(self.dO), P(self.lse), P(self.D), P(self.acc),
                P(self.dq), P(self.dk), P(self.dv), P(self.part), self.splits, B, H, self.Hkv, N,
                d, int(causal), scale, s), "attn_bwd_gqa_split")
        else:
            self.attn.attn_bwd(P(self.q), P(self.k), P(self.v), P(self.dO), P(self.lse), P(self.D),
                               P(self.acc), P(self.dq), P(self.dk), P(self.dv), B, H, N, d, causal,
                               scale, s, Hkv=self.Hkv)

    def train_step(self, s, ev=None, stream=None):
        """attn_fwd_train + attn_bwd_preprocess_o32 + attn_bwd; events between."""
        P = lambda t: t.data_ptr()
        B, H, N, d, causal, scale = self._args()
        if ev:
            ev[0].record(stream)
        self.attn.attn_fwd_train(P(self.q), P(self.k), P(self.v), P(self.o), P(self.o32),
                                 P(self.lse), B, H, N, d, causal, scale, s, Hkv=self.Hkv)
        if ev:
            ev[1].record(stream)
        self.attn.attn_bwd_preprocess_o32(P(self.o32), P(self.dO), P(self.D), P(self.acc), B, H,
                                          N, d, s)
        if ev:
            ev[2].record(stream)
        self.bwd_main(s)
        if ev:
            ev[3].record(stream)

    def exact_step(self, s, ev=None, stream=None):
        """attn_fwd + attn_bwd_preprocess (D from recomputed P and dP) + attn_bwd."""
        P = lambda t: t.data_ptr()
        B, H, N, d, causal, scale = self._args()
        if ev:
            ev[0].record(stream)
        self.fwd(s)
        if ev:
            ev[1].record(stream)
        self.attn.attn_bwd_preprocess(P(self.q), P(self.k), P(self.v), P(self.dO), P(self.lse),
                                      P(self.D), P(self.acc), B, H, N, d, causal, scale, s,
                                      Hkv=self.Hkv)
        if ev:
            ev[2].record(stream)
        self.bwd_main(s)
        if ev:
            ev[3].record(stream)


def _mean(xs):
    return sum(xs) / len(xs)


def _workload_entry(w, dev, stream, flush, steps, warmup, peaks, with_cpu):
    """Compact measurement of one more workload for the JSON line: the
    training step (fwd+bwd workloads) or the forward (forward-only
    workload, as latency), its roofline and a CPU sample of the oracle."""
    import torch
    prob = _Problem(w, dev)
    s = int(stream.cuda_stream)
    peak = peaks["bf16_tflops"]
    fevs = _timed_steps(stream, flush, lambda ev: (ev and ev[0].record(stream), prob.fwd(s),
                                                   ev and ev[1].record(stream)), steps, warmup, 2)
    t_fwd = [e[0].elapsed_time(e[1]) for e in fevs]
    ms_fwd = _mean(t_fwd)
    entry = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
             "qk_mult": w.qk_mult, "seed": w.seed}
    if not w.backward:
        p = _percentiles(t_fwd)
        entry.update({
            "pass": "fwd", "latency_us_p10_p50_p90": [round(1000 * x, 2) for x in p],
            "fwd_tflops": round(w.flops_fwd() / (p[1] * 1e-3) / 1e12, 3),
            "roofline": {"kernel": "attn_fwd", "bound": "latency (%d CTAs for 152 SMs)" % (
                w.B * w.H * ((w.N + 255) // 256)), "achieved": round(w.flops_fwd() / (p[1] * 1e-3) / 1e12, 3),
                "peak": peak, "unit": "TFLOP/s", "frac": round(w.flops_fwd() / (p[1] * 1e-3) / 1e12 / peak, 5)}})
    else:
        evs = _timed_steps(stream, flush, lambda ev: prob.train_step(s, ev, stream), steps, warmup, 4)
        t_step = [e[0].elapsed_time(e[3]) for e in evs]
        ms_step = _mean(t_step)
        ms_bwd = _mean([e[2].elapsed_time(e[3]) for e in evs])
        xevs = _timed_steps(stream, flush, lambda ev: prob.exact_step(s, ev, stream), steps, warmup, 4)
        ms_exact = _mean([e[0].elapsed_time(e[3]) for e in xevs])
        ms_exact_pre = _mean([e[1].elapsed_time(e[2]) for e in xevs])
        fb = w.flops_fwd_bwd()
        # the backward kernel's algorithmic work: 5 MMAs x 2 N^2 d per head
        # (S and dP recomputed, dV, dK, dQ), halved for causal
        bwd_flops = 10.0 * w.B * w.H * w.N * w.N * w.d / (2 if w.causal else 1)
        entry.update({
            "pass": "fwd+bwd", "ms_per_step": round(ms_step, 4),
            "tflops": round(fb / (ms_step * 1e-3) / 1e12, 2),
            "frac_of_peak": round(fb / (ms_step * 1e-3) / 1e12 / peak, 4),
            "fwd_ms": round(ms_fwd, 4), "fwd_tflops": round(w.flops_fwd() / (ms_fwd * 1e-3) / 1e12, 2),
            "fwd_frac_of_peak": round(w.flops_fwd() / (ms_fwd * 1e-3) / 1e12 / peak, 4),
            "fwd_train_ms": round(_mean([e[0].elapsed_time(e[1]) for e in evs]), 4),
            "bwd_preprocess_o32_ms": round(_mean([e[1].elapsed_time(e[2]) for e in evs]), 4),
            "step_exact_d_ms": round(ms_exact, 4), "bwd_preprocess_exact_d_ms": round(ms_exact_pre, 4),
            "roofline": {"kernel": "attn_bwd (main kernel + dQ convert)", "bound": "tensor",
                         "achieved": round(bwd_flops / (ms_bwd * 1e-3) / 1e12, 2), "peak": peak,
                         "unit": "TFLOP/s",
                         "frac": round(bwd_flops / (ms_bwd * 1e-3) / 1e12 / peak, 4)}})
    if torch.cuda.is_available() and prob.attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during workload %s" % w.name)
    if with_cpu:
        entry["cpu_baseline"] = cpu_sample(w, prob.x)
    del prob
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    import io_aware_exact_gb300 as attn

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    w = WORKLOADS[args.workload]
    B, H, N, d, causal = w.B, w.H, w.N, w.d, w.causal
    Hkv = args.kv_heads or H
    if H % Hkv != 0:
        raise SystemExit("--kv-heads must divide the workload's %d heads" % H)
    prob = _Problem(w, dev, rank, Hkv)
    x = prob.x
    q, k, v, dO = prob.q, prob.k, prob.v, prob.dO
    o, lse, o32, D, acc = prob.o, prob.lse, prob.o32, prob.D, prob.acc
    dq, dk, dv = prob.dq, prob.dk, prob.dv
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    s = int(stream.cuda_stream)
    scale = w.scale
    splits = prob.splits

    for _ in range(args.warmup):
        flush.zero_()   # the flush kernel's first launch also happens here, untimed
        prob.train_step(s)
    torch.cuda.synchronize()
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()  # L2 flush between steps, outside the per-step events
            prob.train_step(s, evs[i], stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        wall = time.perf_counter() - t0
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during the timed steps")
    t_step = [e[0].elapsed_time(e[3]) for e in evs]
    t_fwd = [e[0].elapsed_time(e[1]) for e in evs]
    t_pre = [e[1].elapsed_time(e[2]) for e in evs]
    t_bwd = [e[2].elapsed_time(e[3]) for e in evs]
    ms_step = dist_max(sum(t_step) / len(t_step), dev)

    # forward alone (attn_fwd: O and lse, no fp32 O), the inference forward,
    # timed per launch with the same L2 flush between launches
    fevs = _timed_steps(stream, flush, lambda ev: (ev and ev[0].record(stream), prob.fwd(s),
                                                   ev and ev[1].record(stream)),
                        args.steps, 3, 2)
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during the forward-only launches")
    ms_fwd_only = dist_max(statistics.mean(e[0].elapsed_time(e[1]) for e in fevs), dev)

    # the same step with D computed from recomputed P and dP (attn_fwd +
    # attn_bwd_preprocess + attn_bwd, no fp32 O), for comparison
    xevs = _timed_steps(stream, flush, lambda ev: prob.exact_step(s, ev, stream), args.steps, 3, 4)
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during the exact-D steps")
    ms_exact = statistics.mean(e[0].elapsed_time(e[3]) for e in xevs)
    ms_exact_pre = statistics.mean(e[1].elapsed_time(e[2]) for e in xevs)

    # end to end through the public API: pinned host inputs in, results out.
    # Steps are pipelined over two buffer sets and three streams, as a user
    # feeding this API would: step k's inputs go up while step k-1 computes;
    # O and lse come down as soon as the forward has finished, dQ, dK, dV
    # after the backward, while the next step computes.  Every step copies all
    # of its inputs in and all of its results out inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        hx = {kk: vv.pin_memory() for kk, vv in x.items()}
        res = (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        bufs = []
        for _ in range(2):
            b = {"in": {kk: torch.empty_like(vv, device=dev) for kk, vv in x.items()},
                 "out": {n: torch.empty_like(t) for n, t in res},
                 "host": {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in res}}
            for e in ("ev_qkv", "ev_do", "ev_fwd", "ev_comp", "ev_out"):
                b[e] = torch.cuda.Event()
                b[e].record(stream)
            bufs.append(b)
        torch.cuda.synchronize()

        def e2e_step(kstep):
            b = bufs[kstep % 2]
            s_in.wait_event(b["ev_comp"])          # inputs: their last reader is done
            with torch.cuda.stream(s_in):
                for kk in ("q", "k", "v"):
                    b["in"][kk].copy_(hx[kk], non_blocking=True)
                b["ev_qkv"].record(s_in)
                b["in"]["dO"].copy_(hx["dO"], non_blocking=True)
                b["ev_do"].record(s_in)
            stream.wait_event(b["ev_qkv"])
            stream.wait_event(b["ev_out"])         # outputs: their last download is done
            oo, ll, o32_ = attn.forward(b["in"]["q"], b["in"]["k"], b["in"]["v"], causal, scale,
                                        o=b["out"]["o"], lse=b["out"]["lse"], o32=o32, stream=stream)
            b["ev_fwd"].record(stream)
            stream.wait_event(b["ev_do"])
            attn.backward(b["in"]["q"], b["in"]["k"], b["in"]["v"], oo, ll, b["in"]["dO"], causal, scale,
                          dq=b["out"]["dq"], dk=b["out"]["dk"], dv=b["out"]["dv"], D=D, dq_accum=acc,
                          o32=o32_, stream=stream)
            b["ev_comp"].record(stream)
            s_out.wait_event(b["ev_fwd"])
            with torch.cuda.stream(s_out):
                for n in ("o", "lse"):
                    b["host"][n].copy_(b["out"][n], non_blocking=True)
                s_out.wait_event(b["ev_comp"])
                for n in ("dq", "dk", "dv"):
                    b["host"][n].copy_(b["out"][n], non_blocking=True)
                b["ev_out"].record(s_out)

        for kstep in range(2):
            e2e_step(kstep)
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        s_in.wait_event(ea)
        s_out.wait_event(ea)
        for kstep in range(args.e2e_steps):
            e2e_step(kstep)
        stream.wait_event(bufs[(args.e2e_steps - 1) % 2]["ev_out"])
        eb.record(stream)
        torch.cuda.synchronize()
        if attn.attn_get_device_status() != 0:
            raise RuntimeError("device status set during the end-to-end steps")
        # the downloaded results equal a device-resident step on the same
        # inputs (dQ is summed in no fixed order and is left out)
        ro, rl, r32 = attn.forward(q, k, v, causal, scale, o32=True)
        _, rk, rv = attn.backward(q, k, v, ro, rl, dO, causal, scale, o32=r32)
        torch.cuda.synchronize()
        last = bufs[(args.e2e_steps - 1) % 2]["host"]
        for n, t in (("o", ro), ("lse", rl), ("dk", rk), ("dv", rv)):
            if not torch.equal(last[n], t.cpu()):
                raise RuntimeError("end-to-end result %s differs from the device-resident step" % n)
        del ro, rl, r32, rk, rv, bufs
        ms_e2e = ea.elapsed_time(eb) / args.e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for n, t in res)
        e2e = {"value": round(world * w.flops_fwd_bwd() / (ms_e2e * 1e-3) / 1e12, 2),
               "unit": "TFLOPS", "ms_per_step": round(ms_e2e, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelined": "2 buffer sets; H2D, compute and D2H on separate streams"}

    peaks = _peaks()
    flops_fb = w.flops_fwd_bwd()
    tflops_fb = whole_job_rate(world, flops_fb, ms_step) / 1e12
    ms_fwd = statistics.mean(t_fwd)
    ms_bwd = statistics.mean(t_bwd)
    tflops_fwd = whole_job_rate(world, w.flops_fwd(), ms_fwd_only) / 1e12
    tflops_fwd_train = w.flops_fwd() / (ms_fwd * 1e-3) / 1e12
    # dominant kernel: the backward main kernel (timed with its dQ convert);
    # algorithmic work = 5 MMAs x 2 N^2 d per head, halved for causal
    flops_bwd_kernel = 10.0 * B * H * N * N * d / (2 if causal else 1)
    bwd_tflops = flops_bwd_kernel / (ms_bwd * 1e-3) / 1e12
    # One denominator for every fraction: the burst bf16 peak.  The timed
    # regions are tens of milliseconds at full SM clock, the regime the burst
    # figure was measured in; the sustained figure (seconds under the power
    # cap, at a lower clock) is given beside the step's fraction, labelled.
    peak_sus = peaks["bf16_tflops_sustained"]
    peak_burst = peaks["bf16_tflops"]
    # the committed ncu summary is of the multi-head headline workload
    traffic = profile_traffic(args.workload) if Hkv == H else None
    workload = args.workload if Hkv == H else "%s_gqa_kv%d" % (args.workload, Hkv)
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(tflops_fb, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), Q and K x3, bf16)",
        "config": {"workload": workload, "B": B, "H": H, "kv_heads": Hkv, "gqa_splits": splits,
                   "N": N, "d": d,
                   "causal": causal,
                   "global_batch": B * world, "seq_len": N,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs 268 MB > 126 MB L2, and L2 flushed (252 MB write) between steps",
                   "flop_convention": "fwd 4BHN^2d, fwd+bwd 10BHN^2d, halved for causal"},
        "frac_of_peak": round(tflops_fb / peak_burst, 4),
        "peak": peak_burst, "peak_kind": "bf16 burst, %s" % peaks["source"],
        "frac_of_sustained_peak": round(tflops_fb / peak_sus, 4),
        "fwd": {"kernel": "attn_fwd (O, lse)", "tflops": round(tflops_fwd, 2),
                "ms": round(ms_fwd_only, 4), "frac_of_peak": round(tflops_fwd / peak_burst, 4),
                "peak": peak_burst, "peak_kind": "bf16 burst, %s" % peaks["source"]},
        "fwd_train": {"kernel": "attn_fwd_train (O, fp32 O, lse), inside the step",
                      "tflops": round(tflops_fwd_train, 2), "ms": round(ms_fwd, 4)},
        "fwd_bwd_14x_tflops": round(world * 14.0 * B * H * N * N * d / (2 if causal else 1)
                                    / (ms_step * 1e-3) / 1e12, 2),
        "bwd_preprocess_ms": round(statistics.mean(t_pre), 4),
        "step_exact_d": {"path": "attn_fwd + attn_bwd_preprocess (D from recomputed P, dP) + attn_bwd",
                         "ms": round(ms_exact, 4), "preprocess_ms": round(ms_exact_pre, 4),
                         "tflops": round(flops_fb / (ms_exact * 1e-3) / 1e12, 2)},
        "roofline": {"kernel": "attn_bwd (main kernel + dQ convert)", "bound": "tensor",
                     "achieved": round(bwd_tflops, 2), "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": round(bwd_tflops / peak_burst, 4), "traffic": traffic,
                     "peak_kind": "bf16 burst, %s" % peaks["source"]},
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
        "step_ms_p10_p50_p90": [round(x, 4) for x in _percentiles(t_step)],
        "seed": w.seed + 100 * rank,
        "env": _environment(dev),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_heads)
    # The other workloads, each timed the same way (fwd+bwd ones as the
    # training step, the forward-only one as per-launch latency), one GPU only.
    if world == 1 and not args.no_workloads and Hkv == H:
        del prob, x, q, k, v, dO, o, lse, o32, D, acc, dq, dk, dv
        torch.cuda.empty_cache()
        line["workloads"] = [
            _workload_entry(WORKLOADS[n], dev, stream, flush, max(args.steps, 20), args.warmup,
                            peaks, not args.no_cpu_baseline)
            for n in sorted(WORKLOADS, key=lambda n: (WORKLOADS[n].N, WORKLOADS[n].d))
            if n != args.workload]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        import torch.distributed as dist
        dist.destroy_process_group()


BWD_PROFILE = os.path.join(ROOT, "profiles", "attn_bwd_kernel_causal_b2_h16_n8192_d128.md")
BWD_SOURCES = [os.path.join(ROOT, "io_aware_exact_gb300", "csrc", f)
               for f in ("attn_bwd.cu", "attn_common.cuh", "ptx.cuh")]


def kernel_source_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for p in BWD_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(workload):
    """DRAM bytes per launch of the backward main kernel from the committed ncu
    summary, or None if there is none for this workload or the kernel's source
    changed since it was captured."""
    if workload != HEADLINE or not os.path.exists(BWD_PROFILE):
        return None
    fields = {}
    with open(BWD_PROFILE) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256") != kernel_source_sha256():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _percentiles(xs, qs=(0.1, 0.5, 0.9)):
    """Nearest-rank percentiles of a list of times."""
    ys = sorted(xs)
    return [ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))] for q in qs]


def _environment(dev):
    """Device, driver and library versions for the JSON line."""
    import torch
    import io_aware_exact_gb300 as attn
    prop = torch.cuda.get_device_properties(dev)
    env = {"gpu": prop.name, "sm_count": prop.multi_processor_count,
           "cc": "%d.%d" % (prop.major, prop.minor), "torch": torch.__version__,
           "cuda_runtime": torch.version.cuda, "library": attn.version()}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], capture_output=True, text=True, timeout=20)
        env["driver"] = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        env["driver"] = None
    return env


def _oracle_step(w, x, heads):
    """Oracle forward + backward of the given (b, h) heads; returns seconds."""
    import numpy as np
    import oracle
    f = lambda t: t.float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    for (b, h) in heads:
        qh, kh, vh, dOh = (f(x[n][b, h]) for n in ("q", "k", "v", "dO"))
        oracle.attention_forward(qh, kh, vh, w.causal, w.scale)
        oracle.attention_backward(qh, kh, vh, dOh, w.causal, w.scale)
    return time.perf_counter() - t0


def cpu_baseline(w, nheads):
    import oracle
    oracle.build()
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    heads = [(0, h) for h in range(min(nheads, w.H))]
    secs = _oracle_step(w, x, heads)
    per_head = w.flops_fwd_bwd() / (w.B * w.H)
    return {"value": round(per_head * len(heads) / secs / 1e12, 6), "unit": "TFLOPS",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d of %d heads (b=0), all rows, fwd+bwd, %.1f s" % (
                len(heads), w.B * w.H, secs)}


def cpu_sample(w, x=None):
    """The oracle on a bounded sample of workload w, in the graded FLOP
    convention: whole heads while they take under ~2 s (all rows, fwd and,
    for training workloads, bwd), else 128 query rows and 128 key columns of
    head (0, 0) with the most visible pairs."""
    import numpy as np
    import oracle
    oracle.build()
    if x is None:
        x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_grad=True)
    per_head = (w.flops_fwd_bwd() if w.backward else w.flops_fwd()) / (w.B * w.H)
    if per_head < 2e10:
        heads = [(0, h) for h in range(min(w.H, max(1, int(4e10 // per_head))))]
        f = lambda t: t.float().numpy().astype(np.float64)
        t0 = time.perf_counter()
        for (b, h) in heads:
            qh, kh, vh, dOh = (f(x[n][b, h]) for n in ("q", "k", "v", "dO"))
            oracle.attention_forward(qh, kh, vh, w.causal, w.scale)
            if w.backward:
                oracle.attention_backward(qh, kh, vh, dOh, w.causal, w.scale)
        secs = time.perf_counter() - t0
        return {"value": round(per_head * len(heads) / secs / 1e12, 6), "unit": "TFLOPS",
                "cores": oracle.num_threads(), "kind": "oracle",
                "sample": "%d of %d heads, all rows, %s, %.2f s" % (
                    len(heads), w.B * w.H, "fwd+bwd" if w.backward else "fwd", secs)}
    n = 128
    rows = np.arange(w.N - n, w.N, dtype=np.int64)
    cols = np.arange(0, n, dtype=np.int64)
    f = lambda t: t.float().numpy().astype(np.float64)
    qh, kh, vh, dOh = (f(x[nm][0, 0]) for nm in ("q", "k", "v", "dO"))
    lse_all, D_all, _ = oracle.attention_backward_rows(qh, kh, vh, dOh, w.causal, w.scale,
                                                       with_dq=False)
    secs = _ref_sample(w, x, rows, cols, lse_all, D_all)
    pairs = (float(np.sum(rows + 1)) + float(np.sum(w.N - cols))) if w.causal else 2.0 * n * w.N
    return {"value": round(10.0 * w.d * pairs / 2.0 / secs / 1e12, 6), "unit": "TFLOPS",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "head (0,0): last %d query rows and first %d key columns, fwd+bwd, %.2f s" % (
                n, n, secs)}


def _ref_sample(w, x, rows, cols, lse_all, D_all):
    """One reference step: the oracle's forward and backward row passes over
    `rows` and its backward column pass over `cols` of head (0, 0)."""
    import numpy as np
    import oracle
    f = lambda t: t.float().numpy().astype(np.float64)
    qh, kh, vh, dOh = (f(x[n][0, 0]) for n in ("q", "k", "v", "dO"))
    t0 = time.perf_counter()
    oracle.attention_forward(qh, kh, vh, w.causal, w.scale, rows=rows)
    oracle.attention_backward_rows(qh, kh, vh, dOh, w.causal, w.scale, rows=rows)
    oracle.attention_backward_cols(qh, kh, vh, dOh, lse_all, D_all, w.causal, w.scale, cols=cols)
    return time.perf_counter() - t0


def run_varlen(args):
    """The training step (forward with fp32 O, D preprocess, backward) on a
    packed variable-length batch: 32 sequences, lengths drawn uniformly from
    [256, 8192] (seeded), H = 16, d = 128, causal, Q and K x3.  FLOPs count
    only the real tokens: sum over sequences of 10 H L^2 d / 2, no padding."""
    import torch
    import numpy as np
    import io_aware_exact_gb300 as attn
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(1234)
    lengths = rng.integers(256, 8193, size=32)
    H, d = 16, 128
    Hkv = args.kv_heads or H
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    total, max_s = int(cu[-1]), int(lengths.max())
    g = torch.Generator(device="cpu")
    g.manual_seed(4321)
    mk = lambda h, m: (torch.randn((total, h, d), generator=g) * m).to(torch.bfloat16).to(dev)
    q, k, v, dO = mk(H, 3.0), mk(Hkv, 3.0), mk(Hkv, 1.0), mk(H, 1.0)
    cu_d = torch.from_numpy(cu).to(dev)
    scale = d ** -0.5
    o = torch.empty_like(q)
    o32 = torch.empty((total, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((len(lengths), H, max_s), dtype=torch.float32, device=dev)
    D = torch.empty((total, H), dtype=torch.float32, device=dev)
    acc = torch.empty((total, H, d), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(mid=None):
        attn.forward_varlen(q, k, v, cu_d, max_s, True, scale, o=o, lse=lse, o32=o32, stream=stream)
        if mid is not None:
            mid.record(stream)
        attn.backward_varlen(q, k, v, o32, lse, dO, cu_d, max_s, True, scale, dq=dq, dk=dk, dv=dv,
                             D=D, dq_accum=acc, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(evs[i][2])
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during the varlen steps")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms_fwd = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
    flops = float(sum(10.0 * H * int(L) * int(L) * d / 2 for L in lengths))
    padded = 10.0 * H * len(lengths) * max_s * max_s * d / 2
    peak = _peaks().get("bf16_tflops_sustained")
    print(json.dumps({
        "metric": "attention TFLOPS fwd+bwd, packed variable-length batch (real tokens only)",
        "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1), Q and K x3)",
        "config": {"workload": "varlen_causal_32seq_len256to8192_h16_d128", "sequences": len(lengths),
                   "total_tokens": total, "max_seqlen": max_s, "H": H, "kv_heads": Hkv, "d": d,
                   "causal": True, "padding_flops_avoided": round(1 - flops / padded, 3),
                   "l2": "L2 flushed (512 MB write) between steps"},
        "frac_of_peak": round(flops / (ms * 1e-3) / 1e12 / peak, 4) if peak else None,
        "fwd_train_ms": round(ms_fwd, 4), "fwd_train_tflops": round(0.4 * flops / (ms_fwd * 1e-3) / 1e12, 2),
        "bwd_ms": round(ms - ms_fwd, 4), "bwd_tflops": round(0.6 * flops / ((ms - ms_fwd) * 1e-3) / 1e12, 2),
        "clocks": clk.summary(),
    }))


def run_varlen_qk(args):
    """The training step on a packed batch whose keys have lengths of their
    own: 32 sequences, each with Lq query tokens (uniform in [256, 2048]) that
    attend, causally and aligned bottom-right, to Lk = Lq + a cached prefix
    (uniform in [0, 6144]) keys; H = 16, d = 128, Q and K x3 (seeded).  FLOPs
    count only the visible (query, key) pairs, 10 d per pair (the dense
    causal step is 10 B H N^2 d / 2 in the same convention)."""
    import torch
    import numpy as np
    import io_aware_exact_gb300 as attn
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(2468)
    lq = rng.integers(256, 2049, size=32)
    lk = lq + rng.integers(0, 6145, size=32)
    H, d = 16, 128
    Hkv = args.kv_heads or H
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    tq, tk, max_q, max_k = int(cu_q[-1]), int(cu_k[-1]), int(lq.max()), int(lk.max())
    g = torch.Generator(device="cpu")
    g.manual_seed(8642)
    mk = lambda n, h, m: (torch.randn((n, h, d), generator=g) * m).to(torch.bfloat16).to(dev)
    q, k, v, dO = mk(tq, H, 3.0), mk(tk, Hkv, 3.0), mk(tk, Hkv, 1.0), mk(tq, H, 1.0)
    cq, ck = torch.from_numpy(cu_q).to(dev), torch.from_numpy(cu_k).to(dev)
    scale = d ** -0.5
    o = torch.empty_like(q)
    o32 = torch.empty((tq, H, d), dtype=torch.float32, device=dev)
    lse = torch.empty((len(lq), H, max_q), dtype=torch.float32, device=dev)
    D = torch.empty((tq, H), dtype=torch.float32, device=dev)
    acc = torch.empty((tq, H, d), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev):
        if ev:
            ev[0].record(stream)
        attn.forward_varlen(q, k, v, cq, max_q, True, scale, o=o, lse=lse, o32=o32, stream=stream,
                            cu_seqlens_k=ck, max_seqlen_k=max_k)
        if ev:
            ev[2].record(stream)
        attn.backward_varlen(q, k, v, o32, lse, dO, cq, max_q, True, scale, dq=dq, dk=dk, dv=dv,
                             D=D, dq_accum=acc, stream=stream, cu_seqlens_k=ck, max_seqlen_k=max_k)
        if ev:
            ev[1].record(stream)

    with ClockSampler(0) as clk:
        evs = _timed_steps(stream, flush, step, args.steps, args.warmup, 3)
    if attn.attn_get_device_status() != 0:
        raise RuntimeError("device status set during the steps")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms_fwd = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
    # visible pairs of a sequence: query i sees keys 0 .. i + Lk - Lq
    pairs = float(sum(int(a) * (int(b) - int(a)) + int(a) * (int(a) + 1) // 2 for a, b in zip(lq, lk)))
    flops = 10.0 * d * H * pairs
    peak = _peaks().get("bf16_tflops")
    print(json.dumps({
        "metric": "attention TFLOPS fwd+bwd, packed batch with keys of their own lengths (visible pairs only)",
        "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1), Q and K x3)",
        "config": {"workload": "varlen_qk_causal_32seq_q256to2048_prefix0to6144_h16_d128",
                   "sequences": len(lq), "total_q": tq, "total_k": tk, "max_seqlen_q": max_q,
                   "max_seqlen_k": max_k, "H": H, "kv_heads": Hkv, "d": d,
                   "causal": "bottom-right", "l2": "L2 flushed (252 MB write) between steps"},
        "frac_of_peak": round(flops / (ms * 1e-3) / 1e12 / peak, 4) if peak else None,
        "fwd_train_ms": round(ms_fwd, 4), "bwd_ms": round(ms - ms_fwd, 4),
        "clocks": clk.summary(),
    }))


def run_bsparse(args):
    """The training step (forward with fp32 O, D preprocess, backward) with a
    block-sparse layout on the causal B=2 H=16 N=8192 d=128 shape (Q and K
    x3): a seeded random mask per head keeping each 128 x 128 tile with
    probability --bsparse, the diagonal tiles always kept.  FLOPs count only
    the (query, key) pairs the kept tiles leave visible, 10 d per pair (the
    dense causal step is 10 B H N^2 d / 2 in the same convention); the dense
    step on the same inputs is timed beside it."""
    import torch
    import numpy as np
    import io_aware_exact_gb300 as attn
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = WORKLOADS[HEADLINE]
    B, H, N, d = w.B, w.H, w.N, w.d
    nb = (N + 127) // 128
    rng = np.random.default_rng(4321)
    mask = (rng.random((B, H, nb, nb)) < args.bsparse).astype(np.uint8)
    mask[:, :, np.arange(nb), np.arange(nb)] = 1
    rows = np.minimum(128, N - 128 * np.arange(nb))
    full = np.outer(rows, rows).astype(np.float64)
    vis = np.tril(full, -1) + np.diag(rows * (rows + 1) / 2.0)      # causal visible pairs
    pairs = float((mask * vis[None, None]).sum())
    flops = 10.0 * d * pairs
    kept = float((mask * (vis > 0)[None, None]).sum() / ((vis > 0).sum() * B * H))
    x = {n: t.to(dev) for n, t in make_inputs(B, H, N, d, seed=w.seed, qk_mult=w.qk_mult).items()}
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    m = torch.from_numpy(mask).to(dev)
    scale = d ** -0.5
    o = torch.empty_like(q)
    o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    D = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def sparse_step(mid):
        attn.forward_bsparse(q, k, v, m, True, scale, o=o, lse=lse, o32=o32, stream=stream)
        mid.record(stream)
        attn.backward_bsparse(q, k, v, o32, lse, dO, m, True, scale, dq=dq, dk=dk, dv=dv, D=D,
                              dq_accum=acc, stream=stream)

    def dense_step(mid):
        attn.forward(q, k, v, True, scale, o=o, lse=lse, o32=o32, stream=stream)
        mid.record(stream)
        attn.backward(q, k, v, None, lse, dO, True, scale, dq=dq, dk=dk, dv=dv, D=D,
                      dq_accum=acc, stream=stream, o32=o32)

    def timed(step):
        for _ in range(args.warmup):
            step(torch.cuda.Event())
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(evs[i][2])
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if attn.attn_get_device_status() != 0:
            raise RuntimeError("device status set during the block-sparse steps")
        return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                statistics.mean(e[0].elapsed_time(e[2]) for e in evs))

    with ClockSampler(0) as clk:
        ms, ms_fwd = timed(sparse_step)
        ms_dense, _ = timed(dense_step)
    peak = _peaks().get("bf16_tflops_sustained")
    value = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": "attention TFLOPS fwd+bwd, block-sparse layout (kept pairs only)",
        "value": round(value, 2), "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), Q and K x3)",
        "config": {"workload": "bsparse_causal_b2_h16_n8192_d128", "B": B, "H": H, "N": N, "d": d,
                   "causal": True, "tile": 128, "keep_probability": args.bsparse,
                   "kept_tile_fraction": round(kept, 4), "mask": "seeded random per head, diagonal kept",
                   "l2": "L2 flushed (512 MB write) between steps"},
        "frac_of_peak": round(value / peak, 4) if peak else None,
        "fwd_train_ms": round(ms_fwd, 4), "bwd_ms": round(ms - ms_fwd, 4),
        "dense_step_ms": round(ms_dense, 4), "speedup_vs_dense": round(ms_dense / ms, 3),
        "clocks": clk.summary(),
    }))


def run_ring(args):
    """Ring attention emulated on one GPU: the causal B=2 H=16 N=8192 d=128
    training step (Q and K x3) with the sequence split into --ring chunks,
    every (query chunk, key chunk) pair run by the library's kernels and the
    partial results merged (attn_merge) and accumulated (attn_accumulate) as
    a ring of that many devices would.  FLOPs as for the dense causal step;
    the dense step on the same inputs is timed beside it, so the difference
    is what splitting into chunks costs on one device."""
    import torch
    import io_aware_exact_gb300 as attn
    from io_aware_exact_gb300 import ring
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = WORKLOADS[HEADLINE]
    B, H, N, d, R = w.B, w.H, w.N, w.d, args.ring
    if N % R or (N // R) % 8:
        raise SystemExit("--ring must split N into equal chunks")
    x = {n: t.to(dev) for n, t in make_inputs(B, H, N, d, seed=w.seed, qk_mult=w.qk_mult).items()}
    ch = {n: [c.contiguous() for c in torch.chunk(t, R, dim=2)] for n, t in x.items()}
    scale = d ** -0.5
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def ring_step():
        o, lse, o32 = ring.ring_forward(ch["q"], ch["k"], ch["v"], True, scale)
        ring.ring_backward(ch["q"], ch["k"], ch["v"], o32, lse, ch["dO"], True, scale)

    def dense_step():
        o, lse, o32 = attn.forward(x["q"], x["k"], x["v"], True, scale, o32=True)
        attn.backward(x["q"], x["k"], x["v"], None, lse, x["dO"], True, scale, o32=o32)

    def timed(step):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if attn.attn_get_device_status() != 0:
            raise RuntimeError("device status set during the ring steps")
        return statistics.mean(e[0].elapsed_time(e[1]) for e in evs)

    with ClockSampler(0) as clk:
        ms = timed(ring_step)
        ms_dense = timed(dense_step)
    flops = 10.0 * B * H * N * N * d / 2
    peak = _peaks().get("bf16_tflops_sustained")
    value = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": "attention TFLOPS fwd+bwd, ring attention emulated on one GPU",
        "value": round(value, 2), "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), Q and K x3)",
        "config": {"workload": "ring_causal_b2_h16_n8192_d128", "chunks": R, "chunk_len": N // R,
                   "l2": "L2 flushed (512 MB write) between steps"},
        "frac_of_peak": round(value / peak, 4) if peak else None,
        "dense_step_ms": round(ms_dense, 4), "ring_over_dense": round(ms / ms_dense, 3),
        "clocks": clk.summary(),
    }))


def run_dropout(args):
    """The causal B=2 H=16 N=8192 d=128 training step (Q and K x3) with
    dropout p = --dropout on the attention probabilities: the mask is
    regenerated in the forward and the backward from (seed, offset), a new
    offset every step.  FLOPs as for the dense causal step; the step without
    dropout on the same inputs is timed beside it."""
    import torch
    import io_aware_exact_gb300 as attn
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = WORKLOADS[HEADLINE]
    B, H, N, d = w.B, w.H, w.N, w.d
    x = {n: t.to(dev) for n, t in make_inputs(B, H, N, d, seed=w.seed, qk_mult=w.qk_mult).items()}
    q, k, v, dO = x["q"], x["k"], x["v"], x["dO"]
    scale = d ** -0.5
    o = torch.empty_like(q)
    o32 = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    D = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    seed = 0x5EED

    def drop_step(i, mid):
        attn.forward_dropout(q, k, v, args.dropout, seed, i, True, scale, o=o, lse=lse, o32=o32,
                             stream=stream)
        mid.record(stream)
        attn.backward_dropout(q, k, v, o32, lse, dO, args.dropout, seed, i, True, scale, dq=dq,
                              dk=dk, dv=dv, D=D, dq_accum=acc, stream=stream)

    def plain_step(i, mid):
        attn.forward(q, k, v, True, scale, o=o, lse=lse, o32=o32, stream=stream)
        mid.record(stream)
        attn.backward(q, k, v, None, lse, dO, True, scale, dq=dq, dk=dk, dv=dv, D=D,
                      dq_accum=acc, stream=stream, o32=o32)

    def timed(step):
        for i in range(args.warmup):
            step(i, torch.cuda.Event())
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(args.warmup + i, evs[i][2])
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        if attn.attn_get_device_status() != 0:
            raise RuntimeError("device status set during the dropout steps")
        return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
                statistics.mean(e[0].elapsed_time(e[2]) for e in evs))

    with ClockSampler(0) as clk:
        ms, ms_fwd = timed(drop_step)
        ms_plain, ms_plain_fwd = timed(plain_step)
    flops = 10.0 * B * H * N * N * d / 2
    peak = _peaks().get("bf16_tflops_sustained")
    value = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": "attention TFLOPS fwd+bwd with dropout on P",
        "value": round(value, 2), "unit": "TFLOPS", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), Q and K x3)",
        "config": {"workload": "dropout_causal_b2_h16_n8192_d128", "p_drop": args.dropout,
                   "l2": "L2 flushed (512 MB write) between steps"},
        "frac_of_peak": round(value / peak, 4) if peak else None,
        "fwd_train_ms": round(ms_fwd, 4), "bwd_ms": round(ms - ms_fwd, 4),
        "no_dropout_step_ms": round(ms_plain, 4), "no_dropout_fwd_train_ms": round(ms_plain_fwd, 4),
        "clocks": clk.summary(),
    }))


def run_reference(args):
    """The fp64 CPU oracle, as it stands, timed on the host cores.

    A step is a bounded sample of the workload: for head (0, 0), the last
    256 query rows (forward + backward row pass) and the first 256 key
    columns (backward column pass); those are the rows/columns with the most
    visible (query, key) pairs under the causal mask.  Its FLOPs in the stated
    convention are 10*d per visible pair, averaged over the row-side and
    column-side pairs processed (for a whole head both equal N^2/2, giving
    10*N^2*d/2).  The column pass needs every row's lse and D, which the
    oracle computes once before timing.
    """
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    w = WORKLOADS[args.workload]
    x = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    n = min(256, w.N)
    rows = np.arange(w.N - n, w.N, dtype=np.int64)
    cols = np.arange(0, n, dtype=np.int64)
    f = lambda t: t.float().numpy().astype(np.float64)
    qh, kh, vh, dOh = (f(x[nm][0, 0]) for nm in ("q", "k", "v", "dO"))
    lse_all, D_all, _ = oracle.attention_backward_rows(qh, kh, vh, dOh, w.causal, w.scale,
                                                       with_dq=False)
    if w.causal:
        row_pairs = float(np.sum(rows + 1))
        col_pairs = float(np.sum(w.N - cols))
    else:
        row_pairs = col_pairs = float(n * w.N)
    flops = 10.0 * w.d * (row_pairs + col_pairs) / 2.0
    for _ in range(args.warmup):
        _ref_sample(w, x, rows, cols, lse_all, D_all)
    times = [_ref_sample(w, x, rows, cols, lse_all, D_all) for _ in range(args.steps)]
    ms = 1000.0 * sum(times) / len(times)
    value = round(flops / (ms * 1e-3) / 1e12, 6)
    sample = ("head (0,0): last %d query rows (fwd + bwd row pass) and first %d key columns "
              "(bwd column pass) per step" % (n, n))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, bf16 values)",
            "config": {"workload": args.workload, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="grouped K/V heads (GQA / MQA): K and V keep only this many heads")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-heads", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the named workload (by default the JSON line also carries "
                         "every other workload's numbers under \"workloads\")")
    ap.add_argument("--varlen", action="store_true",
                    help="time the step on a packed variable-length batch instead")
    ap.add_argument("--varlen-qk", action="store_true",
                    help="time the step on a packed batch whose keys have lengths of their own "
                         "(queries after a cached prefix) instead")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="time the step with dropout of this probability on P instead")
    ap.add_argument("--ring", type=int, default=0,
                    help="time the step as ring attention over this many chunks, emulated "
                         "on one GPU, instead")
    ap.add_argument("--bsparse", type=float, default=0.0,
                    help="time the step with a random block-sparse layout keeping this "
                         "fraction of tiles instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.varlen:
        run_varlen(args)
    elif args.varlen_qk:
        run_varlen_qk(args)
    elif args.bsparse > 0:
        run_bsparse(args)
    elif args.ring > 0:
        run_ring(args)
    elif args.dropout > 0:
        run_dropout(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
