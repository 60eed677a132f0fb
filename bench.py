"""Benchmark: exact tiled attention forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

A step is one pass of the whole hot path over one batch of synthetic input:
attn_fwd (O, LSE) then attn_bwd (D pre-pass, recompute kernel, dQ finalize)
on the workload's tensors, already resident in device memory. The default
workload is the largest configuration that fits one GPU: B=1 H=16 N=32768
d=128 bf16 causal forward + backward (long context, where a materialised
score matrix would need 32 GiB per layer).

Throughput is useful attention FLOPs per second: 4 B H N^2 d per forward,
2.5x that per backward, halved for causal ("FlashAttention", "Checking it on
a real system"). Prints ONE JSON line on rank 0.

Timing: W untimed warm-up steps, then K timed steps between a barrier and a
device synchronize. The default workload's inputs (Q, K, V, dO: 537 MB) are
larger than L2 (129 MB); a 256 MiB buffer is also rewritten before every
step (outside the per-step events), so smaller workloads start cold too.
Each step's fwd and bwd are bracketed by CUDA events on the launching stream.
Under torchrun every rank runs its own replica (weak scaling) and the max
over ranks is reported; nothing crosses ranks except the timing reduction.

--impl reference times the fp64 CPU oracle instead, on a bounded sample of
the same workload, on rank 0's host cores: whole heads when N <= 4096, else
the leading 4096 x 4096 block of each sampled head (query rows and keys
0..4095; for a causal workload exactly those rows' forward and dQ).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s at 1 GB300 and % of dense bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# our kernels per step: forward 1, backward 3 (pre-pass, recompute kernel, dQ finalize)
LAUNCHES_FWD = 1
LAUNCHES_BWD = 3


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def step_flops(w: W.Workload, backward: bool = True) -> float:
    f = W.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    if backward and w.backward:
        f += W.attention_flops(w.B, w.H, w.N, w.d, w.causal, backward=True)
    return f


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.first = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)  # the sampler is running before the timed region starts
            self.first = len(self.lines)
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
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        # samples taken after the timed region began (the last pre-region one included)
        for line in self.lines[max(0, self.first - 1):]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- oracle arm
SAMPLE_ROWS = 4096


def oracle_sample(w: W.Workload, budget_s: float, max_heads=None, inp=None):
    """Time the fp64 oracle (forward + backward) on sampled heads of the workload until the
    budget is used; returns (seconds, flops of the sample, heads, rows per head).

    A sampled head is a whole head when N <= SAMPLE_ROWS, else its leading SAMPLE_ROWS x
    SAMPLE_ROWS block: query rows and keys 0 .. SAMPLE_ROWS-1 of the workload's own tensors.
    For a causal workload those query rows see only those keys, so the block's forward and dQ
    are exactly the workload's; its dK and dV hold those rows' share. FLOPs are counted for
    the block as for a problem of that length (4 n^2 d, x3.5 with the backward, halved for
    causal)."""
    from oracle import ref
    import torch
    n = min(w.N, SAMPLE_ROWS)
    if inp is None:
        inp = W.make_inputs(w, shape=(1, min(w.H, 4), w.N, w.d))
    nh = min(w.H, 4)
    f64 = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    q, k, v = (f64(inp[x][0, :nh, :n]) for x in ("q", "k", "v"))
    do = f64(inp["do"][0, :nh, :n]) if "do" in inp else None
    maskh = None if inp.get("mask") is None else f64(inp["mask"][0, 0, :n, :n])
    t0 = time.perf_counter()
    heads = 0
    while True:
        h = heads % q.shape[0]
        ref.forward_head(q[h], k[h], v[h], w.scale, w.causal, maskh)
        if w.backward and do is not None:
            ref.backward_head(q[h], k[h], v[h], do[h], w.scale, w.causal, maskh)
        heads += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_heads and heads >= max_heads):
            break
    flops = step_flops(W.Workload(**{**w.__dict__, "B": 1, "H": heads, "N": n}))
    return el, flops, heads, n


def _sample_text(w, heads, n, el=None):
    what = "whole head(s)" if n == w.N else f"leading {n} x {n} block(s) of head(s)"
    t = f"{heads} {what} of the workload, fp64 oracle forward+backward"
    return t + (f", {el:.1f} s" if el is not None else "")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    inp = W.make_inputs(w)
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, max_heads=1, inp=inp)
    secs, flops, heads, n = [], [], 0, w.N
    for _ in range(args.steps):
        el, fl, hd, n = oracle_sample(w, args.ref_budget, max_heads=None, inp=inp)
        secs.append(el)
        flops.append(fl)
        heads += hd
    value = sum(flops) / sum(secs) / 1e12
    ms = 1000.0 * sum(secs) / len(secs)
    sample = (f"per step, {_sample_text(w, '', n).strip()} until {args.ref_budget:.0f} s elapsed "
              f"({heads} in {args.steps} steps)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w.describe(), "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- cross-rank bookkeeping
def reduce_max(values, dist=None, device=None):
    """Element-wise max of per-rank timings over all ranks (identity for one rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_rank_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica (weak scaling), timed
    by the slowest rank."""
    return flops_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm
def measure_workload(A, w, steps, warmup, dev, flush):
    """fwd and bwd milliseconds of one workload (CUDA events on the launching
    stream, L2 rewritten before every timed call)."""
    import torch
    inp = W.make_inputs(w)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    mask = inp["mask"].to(dev) if inp.get("mask") is not None else None
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    fwd = lambda: A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse)  # noqa: E731
    calls = [("fwd", fwd)]
    if w.backward:
        do = inp["do"].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(A.bwd_workspace_size(q), 1), dtype=torch.uint8, device=dev)
        bwd = lambda: A.attn_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, mask=mask,  # noqa: E731
                                 dq=dq, dk=dk, dv=dv, workspace=ws)
        calls.append(("bwd", bwd))
    if w.backward and w.d != 256:  # the deterministic backward is built for head dims 64 and 128
        det = lambda: A.attn_bwd_deterministic(q, k, v, o, lse, do, scale=w.scale, causal=w.causal,  # noqa: E731
                                               mask=mask, dq=dq, dk=dk, dv=dv, workspace=ws)
        calls.append(("bwd_deterministic", det))
    for name, fn in calls:
        for _ in range(warmup):
            fwd()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in evs:
            flush.fill_(3)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        res[name] = sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())
    out = {"shape": [w.B, w.H, w.N, w.d], "dtype": w.dtype, "causal": w.causal, "mask": w.mask}
    f = W.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    out["fwd_ms"] = res["fwd"]
    out["fwd_tflops"] = f / (res["fwd"] * 1e-3) / 1e12
    for key in ("bwd", "bwd_deterministic"):  # both counted as 2.5x the forward's FLOPs
        if key in res:
            out[f"{key}_ms"] = res[key]
            out[f"{key}_tflops"] = 2.5 * f / (res[key] * 1e-3) / 1e12
    return out

def measure_fp8(A, w, steps, warmup, dev, flush):
    """FP8 forward milliseconds of one E4M3 workload (CUDA events on the launching stream, L2
    rewritten before every timed call). TFLOP/s counts the same 4 B H N^2 d (halved for causal)
    as the 16-bit forward; the percentage is of the measured bf16 dense peak times the nominal
    E4M3 / bf16 tensor-rate ratio of 2."""
    import torch
    inp = W.make_fp8_inputs(w)
    q, k, v = (inp[n].to(dev).view(torch.float8_e4m3fn) for n in ("q8", "k8", "v8"))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    fn = lambda: A.attn_fwd_fp8(q, k, v, inp["q_ds"], inp["k_ds"], inp["v_ds"], scale=w.scale,  # noqa: E731
                                causal=w.causal, out=o, lse=lse)
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush.fill_(3)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
    f = W.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    return {"shape": [w.B, w.H, w.N, w.d], "dtype": "e4m3", "causal": w.causal, "mask": w.mask, "fwd_ms": ms,
            "fwd_tflops": f / (ms * 1e-3) / 1e12}


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import attn_fwd_03_gb300 as A

    peaks, peak_kind = load_peaks()
    inp = W.make_inputs(w)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    do = inp["do"].to(dev) if w.backward else None
    mask = inp["mask"].to(dev) if inp.get("mask") is not None else None
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq = dk = dv = ws = None
    if w.backward:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(A.bwd_workspace_size(q), 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do) if t is not None)

    def bwd():
        if w.backward:
            A.attn_bwd(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, mask=mask, dq=dq, dk=dk, dv=dv,
                       workspace=ws)

    def step():
        A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse)
        bwd()

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    # events the library records between its three backward launches
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for row in bev:
        for e in row:
            e.record(stream)  # creates the underlying CUDA event
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse)
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    # The per-kernel split of the backward comes from as many further steps, with events
    # recorded between its launches; they stay out of the timed steps above because each
    # event is a stream operation between two kernels that could otherwise overlap.
    if w.backward:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            A.attn_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse)
            A.debug_set_bwd_events(bev[i])
            bwd()
        A.debug_set_bwd_events(None)
        torch.cuda.synchronize()
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    ms = sum(f + b for f, b in zip(fwd_ms, bwd_ms)) / args.steps
    ms_fwd = sum(fwd_ms) / args.steps
    ms_bwd = sum(bwd_ms) / args.steps
    ms_main = ms_pre = ms_fin = 0.0
    if w.backward:
        ms_pre = sum(bev[i][0].elapsed_time(bev[i][1]) for i in range(args.steps)) / args.steps
        ms_main = sum(bev[i][1].elapsed_time(bev[i][2]) for i in range(args.steps)) / args.steps
        ms_fin = sum(bev[i][2].elapsed_time(bev[i][3]) for i in range(args.steps)) / args.steps
    ms, ms_fwd, ms_bwd, ms_pre, ms_main, ms_fin = reduce_max([ms, ms_fwd, ms_bwd, ms_pre, ms_main, ms_fin],
                                                             dist if world > 1 else None, dev)

    f_step = step_flops(w)
    f_fwd = step_flops(w, backward=False)
    value = job_throughput(f_step, world, ms)
    peak = peaks["bf16_tflops"]
    fwd_tflops = f_fwd / (ms_fwd * 1e-3) / 1e12
    bwd_tflops = (f_step - f_fwd) / (ms_bwd * 1e-3) / 1e12 if w.backward else None

    # ---- per-kernel rooflines; the dominant kernel (most time per step) is reported as "roofline"
    peak_src = f"{peak_kind} bf16_tflops (burst: kernels timed inside a step of a few ms)"
    kernels = {"fwd_tc_kernel": {"ms": ms_fwd, "bound": "tensor", "achieved": fwd_tflops, "peak": peak,
                                 "unit": "TFLOP/s", "frac": fwd_tflops / peak}}
    if w.backward:
        main_tflops = (f_step - f_fwd) / (ms_main * 1e-3) / 1e12
        kernels["bwd_tc64_kernel" if w.d == 64 else "bwd_tc_kernel"] = {"ms": ms_main, "bound": "tensor", "achieved": main_tflops, "peak": peak,
                                    "unit": "TFLOP/s", "frac": main_tflops / peak}
        rows = w.B * w.H * w.N
        pre_bytes = rows * w.d * 2 * 2 + rows * w.d * 4 + rows * 2 * 4 + rows * 4
        fin_bytes = rows * w.d * 4 + rows * w.d * 2
        hbm = peaks["hbm_gbs"]
        for name, ms_k, nbytes in (("bwd_prepass_kernel", ms_pre, pre_bytes),
                                   ("bwd_dq_finalize_kernel", ms_fin, fin_bytes)):
            gbs = nbytes / (ms_k * 1e-3) / 1e9 if ms_k > 0 else None
            kernels[name] = {"ms": ms_k, "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                             "frac": gbs / hbm if gbs else None}
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    roof = dict(kernels[dom])
    roof.pop("ms")
    roof.update({"kernel": dom, "traffic": captured_traffic(dom, w.name), "peak_source": peak_src,
                 "note": "achieved = algorithmic FLOPs per launch / CUDA-event launch duration; traffic = "
                         "DRAM bytes per launch from an ncu capture of the same kernel source (null if stale)"})
    if roof.get("bound") == "tensor" and peaks.get("bf16_tflops_sustained"):
        # the timed steps run back to back for seconds under the power cap: the sustained GEMM
        # figure is the other fair denominator (reported beside the burst one, which `frac` uses)
        roof["peak_sustained"] = peaks["bf16_tflops_sustained"]
        roof["frac_of_sustained"] = roof["achieved"] / peaks["bf16_tflops_sustained"]

    # ---- end to end through the public API with pinned host buffers. Every step copies its
    # inputs in and its results out; with two device buffer sets and three streams the copy-in
    # of step i+1 and the copy-out of step i-1 overlap the compute of step i (the copies in the
    # two directions also overlap each other).
    in_names = ("q", "k", "v", "do") if w.backward else ("q", "k", "v")
    h_in = {n: inp[n].pin_memory() for n in in_names}
    h_mask = inp["mask"].pin_memory() if inp.get("mask") is not None else None
    out_names = ("o", "lse", "dq", "dk", "dv") if w.backward else ("o", "lse")
    h_out = {"o": torch.empty_like(inp["q"]).pin_memory(), "lse": torch.empty(q.shape[:3]).pin_memory()}
    if w.backward:
        for n, t in (("dq", inp["q"]), ("dk", inp["k"]), ("dv", inp["v"])):
            h_out[n] = torch.empty_like(t).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values()) + \
        (h_mask.numel() * h_mask.element_size() if h_mask is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    first = {"q": q, "k": k, "v": v, "do": do, "mask": mask, "o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    sets = [first, {n: (torch.empty_like(t) if t is not None else None) for n, t in first.items()}]
    s_cmp, s_in, s_out = stream, torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        b = i & 1
        S = sets[b]
        if i >= 2:
            s_in.wait_event(ev_cmp[b])  # step i-2 has finished reading this set's inputs
        with torch.cuda.stream(s_in):
            for n in in_names:
                S[n].copy_(h_in[n], non_blocking=True)
            if h_mask is not None:
                S["mask"].copy_(h_mask, non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if i >= 2:
            s_cmp.wait_event(ev_out[b])  # step i-2's results have been copied out of this set
        with torch.cuda.stream(s_cmp):
            A.attn_fwd(S["q"], S["k"], S["v"], scale=w.scale, causal=w.causal, mask=S["mask"], out=S["o"],
                       lse=S["lse"])
            if w.backward:
                A.attn_bwd(S["q"], S["k"], S["v"], S["o"], S["lse"], S["do"], scale=w.scale, causal=w.causal,
                           mask=S["mask"], dq=S["dq"], dk=S["dk"], dv=S["dv"], workspace=ws)
            ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for n in out_names:
                h_out[n].copy_(S[n], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    s_in.wait_event(ev_out[(args.steps - 1) & 1])
    e1.record(s_in)
    torch.cuda.synchronize()
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = reduce_max([e2e_ms], dist if world > 1 else None, dev)[0]
    e2e_value = job_throughput(f_step, world, e2e_ms)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**w.describe(), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2" if in_bytes > (129 << 20) else "inputs fit in L2") +
                         "; a 256 MiB buffer is rewritten before every timed step",
                   "step": "attn_fwd + attn_bwd" if w.backward else "attn_fwd"},
        "pct_of_peak": 100.0 * value / world / peak,
        "fwd": {"ms": ms_fwd, "tflops": fwd_tflops, "pct_of_peak": 100.0 * fwd_tflops / peak},
        "bwd": ({"ms": ms_bwd, "tflops": bwd_tflops, "pct_of_peak": 100.0 * bwd_tflops / peak}
                if w.backward else None),
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "pipeline": "pinned host buffers; copy-in, compute and copy-out of consecutive steps overlap "
                            "on three streams with two device buffer sets"},
        "gpu_launches": args.steps * (LAUNCHES_FWD + (LAUNCHES_BWD if w.backward else 0)),
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_all:
        peak = peaks["bf16_tflops"]
        table = {}
        for idx, wk in {**W.WORKLOADS, **W.F16_WORKLOADS, **W.D256_WORKLOADS}.items():
            r = measure_workload(A, wk, 10, 3, dev, flush)
            for key in ("fwd", "bwd", "bwd_deterministic"):
                if f"{key}_tflops" in r and wk.dtype in ("bf16", "f16"):
                    r[f"{key}_pct_of_peak"] = 100.0 * r[f"{key}_tflops"] / peak
            table[wk.name] = r
        for idx, wk in W.FP8_WORKLOADS.items():
            r = measure_fp8(A, wk, 10, 3, dev, flush)
            r["fwd_pct_of_e4m3_peak"] = 100.0 * r["fwd_tflops"] / (2.0 * peak)
            table[wk.name] = r
        for nq in (1, 8):
            table[f"decode_b8_h32_nq{nq}_nk8192_d128_bf16_causal"] = measure_decode(A, dev, peaks["hbm_gbs"], nq)
        line["workloads"] = table
    if world == 1 and not args.no_cpu_baseline:
        el, fl, heads, n = oracle_sample(w, args.cpu_budget, inp=inp)
        line["cpu_baseline"] = {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                                "sample": _sample_text(w, heads, n, el)}
    print(json.dumps(line), flush=True)


def measure_decode(A, dev, hbm_gbs: float, nq: int, B: int = 8, H: int = 32, nk: int = 8192, d: int = 128,
                   steps: int = 20, warmup: int = 3) -> dict:
    """Split-KV decode: nq query rows against an nk-key cache per (b, h). Bound by HBM: the
    algorithmic bytes are K and V read once plus Q, O and LSE. K and V (1 GiB here) exceed L2."""
    import torch
    q = W.random_tensor((B, H, nq, d), 730, torch.bfloat16).to(dev)
    k = W.random_tensor((B, H, nk, d), 731, torch.bfloat16).to(dev)
    v = W.random_tensor((B, H, nk, d), 732, torch.bfloat16).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, nq), dtype=torch.float32, device=dev)
    ws = torch.empty(max(A.decode_workspace_size(q, k, v, causal=True), 1), dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        A.attn_decode(q, k, v, causal=True, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        A.attn_decode(q, k, v, causal=True, out=o, lse=lse, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    if A.attn_status() != A.ATTN_OK:
        raise RuntimeError(A.last_error())
    ms = e0.elapsed_time(e1) / steps
    nbytes = 2 * B * H * nk * d * 2 + 2 * B * H * nq * d * 2 + B * H * nq * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"shape": [B, H, nq, nk, d], "dtype": "bf16", "causal": True, "ms": ms,
            "achieved_gbs": gbs, "pct_of_hbm_peak": 100.0 * gbs / hbm_gbs, "launches": 2,
            "bytes": nbytes}


def captured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from profiles/dram_traffic.json,
    or None when there is no capture or the kernel's sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    for e in doc.get("entries", []):
        if e.get("kernel") != kernel or e.get("workload") != workload:
            continue
        for rel, digest in e.get("sources", {}).items():
            try:
                with open(os.path.join(ROOT, rel), "rb") as f:
                    if hashlib.sha256(f.read()).hexdigest() != digest:
                        return None
            except OSError:
                return None
        return int(e["dram_bytes_read"]) + int(e["dram_bytes_write"])
    return None


def run_table_entry(args):
    """One row of the per-workload table, timed alone on GPU 0 (--steps timed calls after
    --warmup, L2 rewritten before each)."""
    import torch
    import attn_fwd_03_gb300 as A
    every = {**W.WORKLOADS, **W.F16_WORKLOADS, **W.D256_WORKLOADS, **W.FP8_WORKLOADS, **W.PROFILE_WORKLOADS}
    by_name = {wk.name: wk for wk in every.values()}
    if args.table_workload not in by_name:
        raise SystemExit(f"unknown workload {args.table_workload}; one of {sorted(by_name)}")
    wk = by_name[args.table_workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if wk.dtype == "e4m3":
        r = measure_fp8(A, wk, args.steps, args.warmup, dev, flush)
    else:
        r = measure_workload(A, wk, args.steps, args.warmup, dev, flush)
    print(json.dumps({"workload": wk.name, **r}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=5, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=5.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all", action="store_true", help="skip the per-workload forward/backward table")
    ap.add_argument("--decode", type=int, default=None, metavar="NQ",
                    help="time only the split-KV decode entry of the table with NQ query rows "
                         "(B=8 H=32 nk=8192 d=128) and print it as one JSON line")
    ap.add_argument("--table-workload", default=None,
                    help="time only this entry of the per-workload table (a workload name from workloads.py, "
                         "e.g. under a profiler) and print it as one JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.table_workload is not None:
        run_table_entry(args)
        return
    if args.decode is not None:
        import torch
        import attn_fwd_03_gb300 as A
        peaks, _ = load_peaks()
        r = measure_decode(A, torch.device("cuda", 0), peaks["hbm_gbs"], args.decode, steps=args.steps,
                           warmup=args.warmup)
        print(json.dumps({"workload": f"decode_b8_h32_nq{args.decode}_nk8192_d128_bf16_causal", **r}), flush=True)
        return
    w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
