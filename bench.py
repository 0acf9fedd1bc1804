"""Benchmark of the fused attention backward on GB300.

Default workload: GQA backward, B=2, H_q=32, H_k=8, Sq=Sk=8192, D=128, bf16,
causal, non-deterministic dQ reduction, synthetic N(0,1) inputs (seed 3);
O and LSE come from this library's forward.  One step = one attn_bwd call
(preprocess + main + postprocess kernels) over that batch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--deterministic] [--pass bwd|fwd]

Metric: backward TFLOPS = 2.5 * 4 * B * H_q * Sq * Sk * D / t, halved for
causal.  ``--pass fwd`` times the forward (attn_fwd: O and LSE) on the same
workload instead, at 4 * B * H_q * Sq * Sk * D FLOPs (halved for causal).
Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are
independent replicas, one per GPU; value = total FLOPs of all ranks / the
slowest rank's time.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from attention_backward_bwd_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "gqa_b2_hq32_hk8_s8192_d128_bf16_causal"
METRIC = "attention-backward TFLOPS (bf16, 1xGB300) and % of dense tensor-core peak"
METRIC_FWD = "attention-forward TFLOPS (bf16, 1xGB300) and % of dense tensor-core peak"
L2_BYTES = 129 * 2 ** 20


def window_pairs(sq: int, sk: int, causal: bool, window) -> int:
    """Number of (query, key) pairs a local mask allows (bottom-right aligned)."""
    left, right = window
    if causal:
        right = 0
    i = np.arange(sq, dtype=np.int64)
    lo = np.maximum(0, i + (sk - sq) - left) if left >= 0 else np.zeros_like(i)
    hi = np.minimum(sk - 1, i + (sk - sq) + right) if right >= 0 else np.full_like(i, sk - 1)
    return int(np.maximum(0, hi - lo + 1).sum())


def bwd_flops(w: synth.Workload, lengths=None) -> float:
    """2.5 x forward FLOPs (4 B H Sq Sk D), halved when causal; varlen sums sequences.
    With a local window: 10 D FLOPs per allowed (query, key) pair, counted exactly."""
    if w.windowed:
        if w.varlen:
            pairs = sum(window_pairs(n, n, w.causal, w.window) for n in lengths)
        else:
            pairs = w.batch * window_pairs(w.seqlen_q, w.seqlen_k, w.causal, w.window)
        return 10.0 * w.head_dim * w.h_q * pairs
    if w.varlen:
        f = sum(2.5 * 4.0 * w.h_q * n * n * w.head_dim for n in lengths)
    else:
        f = 2.5 * 4.0 * w.batch * w.h_q * w.seqlen_q * w.seqlen_k * w.head_dim
    return f / 2 if w.causal else f


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "src": "fallback"}


def kernel_traffic():
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    valid only while the kernel source still hashes to the profiled version."""
    src = os.path.join(ROOT, "attention_backward_bwd_gb300", "csrc", "bwd_main.cu")
    prof = os.path.join(ROOT, "profiles", "bwd_main_traffic_gqa_b2_hq32_hk8_s8192_d128_causal.txt")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        kv = dict(line.strip().split("=", 1) for line in open(prof) if "=" in line)
        if kv.get("source_sha256_16") == h:
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling (every 50 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"attn_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        load = [s for s, p in zip(sm, pw) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


class DeviceRounds:
    """Device time of rounds of work enqueued from the host.

    Each chunk of rounds is queued behind a device-side sleep that outlasts the
    host's enqueue time for that chunk, so no launch waits for the host and the
    events bracket device time only (on small problems a Python-level call takes
    longer than the kernels it launches).  Chunks keep the launch queue short.
    When the step's resident data would fit in L2 (under twice its size), every
    round first overwrites a buffer of twice the L2 size, outside the events, so
    each timed round starts with a cold L2.
    """

    CHUNK = 32
    SLEEP_HZ = 2.2e9  # cycles per second of the device sleep: at most the SM clock

    def __init__(self, stream, one_round, resident_bytes: int, dev):
        self.stream = stream
        self.flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
                      if resident_bytes < 2 * L2_BYTES else None)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(3):
            if self.flush is not None:
                self.flush.zero_()
            one_round()
        self.host_s = (time.perf_counter() - t0) / 3
        torch.cuda.synchronize()

    def l2_note(self, resident_bytes: int) -> str:
        if self.flush is None:
            return "inputs larger than L2 (%.0f MB resident per step)" % (resident_bytes / 1e6)
        return ("L2 flushed before every timed step (%.0f MB resident per step, %d MB written)"
                % (resident_bytes / 1e6, 2 * L2_BYTES // 2 ** 20))

    def run(self, n: int, body, n_events: int):
        """Runs body(events) n times; `events` holds n_events timing events that
        body records around its stages.  Returns the per-round event lists."""
        rounds = []
        i = 0
        while i < n:
            m = min(self.CHUNK, n - i)
            torch.cuda._sleep(int((1.5 * m * self.host_s + 5e-4) * self.SLEEP_HZ))
            for _ in range(m):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_events)]
                if self.flush is not None:
                    self.flush.zero_()
                body(ev)
                rounds.append(ev)
            i += m
        return rounds


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x: float, dist) -> float:
    """The slowest rank's time: the replicas' job ends when the last one does."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job TFLOP/s of `world` independent replicas: every rank does the
    same work, the job takes as long as the slowest rank."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def run_ours(args):
    import attention_backward_bwd_gb300 as ab
    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    det = bool(args.deterministic or w.deterministic)
    x = synth.make_inputs(w)
    mq = mk = max(x.lengths) if w.varlen else None
    cu_q = x.cu_seqlens_q.to(dev) if w.varlen else None
    cu_k = x.cu_seqlens_k.to(dev) if w.varlen else None
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    window = tuple(w.window) if w.windowed else None
    o, lse = ab.attn_fwd(q, k, v, causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                         max_seqlen_q=mq, max_seqlen_k=mk, window=window, softcap=w.softcap)
    ws = ab.alloc_workspace(q, cu_q, det)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    kw = dict(causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=mq,
              max_seqlen_k=mk, deterministic=det, workspace=ws, dq=dq, dk=dk, dv=dv,
              window=window, softcap=w.softcap)
    stream = torch.cuda.current_stream()
    flops = bwd_flops(w, x.lengths)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, o, do, lse))

    def step():
        ab.attn_bwd(q, k, v, o, lse, do, stream=stream, **kw)

    for _ in range(args.warmup):
        step()
    ab.check_device_status()
    resident = in_bytes + sum(t.numel() * t.element_size() for t in (dq, dk, dv)) + \
        ws.numel() * ws.element_size()
    timer = DeviceRounds(stream, step, resident, dev)

    def whole(ev):
        ev[0].record(stream)
        step()
        ev[1].record(stream)

    def staged(ev):
        ev[0].record(stream)
        ab.attn_bwd(q, k, v, o, lse, do, stream=stream, stage="pre", **kw)
        ev[1].record(stream)
        ab.attn_bwd(q, k, v, o, lse, do, stream=stream, stage="main", **kw)
        ev[2].record(stream)
        ab.attn_bwd(q, k, v, o, lse, do, stream=stream, stage="post", **kw)
        ev[3].record(stream)

    # --- timed region: K steps, device-resident inputs, device time of each step
    torch.cuda.synchronize()
    barrier(dist)
    with ClockSampler(local) as clk:
        steps_ev = timer.run(args.steps, whole, 2)
        torch.cuda.synchronize()
        barrier(dist)
        # per-kernel times over the same number of steps (events on the launch stream)
        evs = timer.run(args.steps, staged, 4)
        torch.cuda.synchronize()
        barrier(dist)
    ab.check_device_status()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in steps_ev)
    ms_max = max_over_ranks(ms, dist)
    t_pre = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_main = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_post = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    # --- end to end: pinned host inputs -> device -> backward -> pinned host results,
    # through attn_bwd_host (padded) or attn_bwd_host_varlen (packed): chunks whose
    # copies overlap the kernels of other chunks.
    hq_ = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in hq_)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    if not w.varlen:
        b_, sq_, hq_n, d_ = q.shape
        hbuf = torch.empty(ab.host_buffer_size(b_, sq_, k.shape[1], hq_n, k.shape[2], d_,
                                               args.chunks), dtype=torch.uint8, device=dev)
        e2e_path = f"attn_bwd_host, chunks={args.chunks or 'auto'}"

        def e2e_step():
            ab.attn_bwd_host(hq_[0], hq_[1], hq_[2], hq_[3], hq_[5], hq_[4], *host_out,
                             causal=w.causal, deterministic=det, chunks=args.chunks,
                             device_buffer=hbuf, stream=stream, window=window,
                             softcap=w.softcap)
    else:
        cu_q_h, cu_k_h = x.cu_seqlens_q.cpu(), x.cu_seqlens_k.cpu()
        need = int(ab.lib().attn_bwd_host_varlen_buffer_size(
            cu_q_h.data_ptr(), cu_k_h.data_ptr(), len(x.lengths), q.shape[0], k.shape[0],
            q.shape[1], k.shape[1], q.shape[2], args.chunks))
        hbuf = torch.empty(need, dtype=torch.uint8, device=dev)
        e2e_path = f"attn_bwd_host_varlen, chunks={args.chunks or 'auto'}"

        def e2e_step():
            ab.attn_bwd_host_varlen(hq_[0], hq_[1], hq_[2], hq_[3], hq_[5], hq_[4], cu_q_h,
                                    cu_k_h, *host_out, causal=w.causal, deterministic=det,
                                    chunks=args.chunks, device_buffer=hbuf, stream=stream,
                                    window=window, softcap=w.softcap)

    for _ in range(2):
        e2e_step()
    barrier(dist)
    n_e2e = max(2, args.steps // 2)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    a1.record(stream)
    barrier(dist)
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / n_e2e, dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peaks = measured_peaks()
    achieved = flops / (t_main * 1e-3) / 1e12
    # The main kernel is timed on its own, a few milliseconds per launch at the
    # clocks recorded below, so its denominator is the burst bf16 GEMM figure
    # (measured the same way); the sustained figure was taken over seconds of
    # back-to-back GEMMs at power-capped clocks and is printed for comparison.
    peak = peaks["bf16_tflops"]
    peak_sus = peaks["bf16_tflops_sustained"]
    traffic = kernel_traffic()
    rows_heads = (sum(x.lengths) if w.varlen else w.batch * w.seqlen_q) * w.h_q
    esz = 2
    pre_bytes = rows_heads * (2 * w.head_dim * esz + 4 + 8 + 4 * w.head_dim)
    post_bytes = rows_heads * (4 * w.head_dim + esz * w.head_dim)
    value = replica_value(flops, ms_max, world)
    cfg = {"workload": w.name, "batch": w.batch if not w.varlen else len(x.lengths),
           "h_q": w.h_q, "h_k": w.h_k, "seqlen": w.seqlen_q if not w.varlen else "varlen",
           "head_dim": w.head_dim, "causal": w.causal, "deterministic": det,
           "l2": timer.l2_note(resident),
           "timing": "device time per step (CUDA events; launches queued ahead of the device)",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if w.varlen:
        cfg["lengths"] = x.lengths
    if w.softcap:
        cfg["softcap"] = w.softcap
    if w.windowed:
        cfg["window"] = list(w.window)
        cfg["flops"] = "10 D per allowed (query, key) pair, counted exactly"
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic N(0,1), seeded; O and LSE from attn_fwd", "config": cfg,
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"bound": "tensor",
                     "kernel": "bwd_main_kernel" if w.head_dim <= 128 else
                               "bwd_wide_kernel (dK/dQ pass + dV pass)",
                     "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_src": "bf16 burst, of " + peaks["src"],
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "traffic": traffic},
        "kernels_ms": {"preprocess": round(t_pre, 4), "main": round(t_main, 4),
                       "postprocess": round(t_post, 4)},
        "hbm": {"preprocess_gbs": round(pre_bytes / (t_pre * 1e-3) / 1e9, 1),
                "postprocess_gbs": round(post_bytes / (t_post * 1e-3) / 1e9, 1),
                "peak_gbs": peaks["hbm_gbs"]},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "path": e2e_path},
        # preprocess, main, postprocess; varlen adds the cu_seqlens check
        "gpu_launches": (4 if w.varlen else 3) * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_budget)
    print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


def run_ours_fwd(args):
    """The forward (attn_fwd) of the workload: O and the natural-log LSE."""
    import attention_backward_bwd_gb300 as ab
    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    mq = mk = max(x.lengths) if w.varlen else None
    cu_q = x.cu_seqlens_q.to(dev) if w.varlen else None
    cu_k = x.cu_seqlens_k.to(dev) if w.varlen else None
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    window = tuple(w.window) if w.windowed else None
    o = torch.empty_like(q)
    lse_shape = (q.shape[1], q.shape[0]) if w.varlen else (q.shape[0], q.shape[2], q.shape[1])
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    kw = dict(causal=w.causal, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=mq,
              max_seqlen_k=mk, window=window, softcap=w.softcap, out=o, lse=lse)
    stream = torch.cuda.current_stream()
    flops = bwd_flops(w, x.lengths) / 2.5
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))

    def step():
        ab.attn_fwd(q, k, v, stream=stream, **kw)

    for _ in range(args.warmup):
        step()
    ab.check_device_status()
    resident = in_bytes + o.numel() * o.element_size() + lse.numel() * lse.element_size()
    timer = DeviceRounds(stream, step, resident, dev)

    def whole(ev):
        ev[0].record(stream)
        step()
        ev[1].record(stream)

    torch.cuda.synchronize()
    barrier(dist)
    with ClockSampler(local) as clk:
        steps_ev = timer.run(args.steps, whole, 2)
        torch.cuda.synchronize()
        barrier(dist)
    ab.check_device_status()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in steps_ev)
    ms_max = max_over_ranks(ms, dist)

    # end to end: pinned host Q, K, V -> device -> attn_fwd -> pinned host O, LSE
    hq_ = [t.cpu().pin_memory() for t in (q, k, v)]
    ho, hl = torch.empty(o.shape, dtype=o.dtype, pin_memory=True), torch.empty(
        lse.shape, dtype=lse.dtype, pin_memory=True)
    dq_, dk_, dv_ = (torch.empty_like(t) for t in (q, k, v))
    h2d = sum(t.numel() * t.element_size() for t in hq_)
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    def e2e_step():
        for dst, src in zip((dq_, dk_, dv_), hq_):
            dst.copy_(src, non_blocking=True)
        ab.attn_fwd(dq_, dk_, dv_, stream=stream, **kw)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier(dist)
    n_e2e = max(2, args.steps // 2)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    a1.record(stream)
    barrier(dist)
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / n_e2e, dist)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peaks = measured_peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    value = replica_value(flops, ms_max, world)
    cfg = {"workload": w.name, "pass": "forward", "batch": w.batch if not w.varlen else len(x.lengths),
           "h_q": w.h_q, "h_k": w.h_k, "seqlen": w.seqlen_q if not w.varlen else "varlen",
           "head_dim": w.head_dim, "causal": w.causal,
           "l2": timer.l2_note(resident),
           "timing": "device time per step (CUDA events; launches queued ahead of the device)",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if w.varlen:
        cfg["lengths"] = x.lengths
    if w.softcap:
        cfg["softcap"] = w.softcap
    if w.windowed:
        cfg["window"] = list(w.window)
    out = {
        "metric": METRIC_FWD, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic N(0,1), seeded", "config": cfg,
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "kernel": "fwd_kernel", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_src": "bf16 burst, of " + peaks["src"], "traffic": None},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "path": "pinned copies + attn_fwd"},
        "gpu_launches": (2 if w.varlen else 1) * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(w, x, n_rows=None):
    """A bounded slice of the workload for the CPU oracle: one query head of
    sequence 0 (one GQA group member), its last ``n_rows`` query rows (all rows
    if None) against every key they see.  With the bottom-right aligned masks
    the last n rows of a sequence are an exact sub-problem (Sq = n, Sk = L), so
    the oracle runs on it unchanged; FLOPs are 10 D per allowed pair of the
    slice (for whole causal heads without a window: the 2.5 x 4 L^2 D / 2
    convention of the GPU line)."""
    from oracle import attn_oracle
    if w.varlen:
        L = x.lengths[0]
        q, k, v, do = x.q[:L], x.k[:L], x.v[:L], x.do[:L]
    else:
        q, k, v, do = x.q[0], x.k[0], x.v[0], x.do[0]
        L = w.seqlen_q
    n = L if n_rows is None else max(1, min(L, int(n_rows)))
    g = w.h_q // w.h_k
    window = tuple(w.window) if w.windowed else None

    def run(h):
        return attn_oracle.head_backward(q[L - n:, h].double().numpy(),
                                         k[:, h // g].double().numpy(),
                                         v[:, h // g].double().numpy(),
                                         do[L - n:, h].double().numpy(), w.scale, w.causal,
                                         window, w.softcap)
    if w.windowed or n < L:
        f_one = 10.0 * w.head_dim * window_pairs(n, L, w.causal, window or (-1, -1))
    else:
        f_one = 2.5 * 4.0 * L * L * w.head_dim / (2 if w.causal else 1)
    return run, f_one, L, n


def cpu_baseline(w, x, budget_s=20.0):
    run, f_one, L, _ = oracle_sample(w, x)
    t0 = time.perf_counter()
    n = 0
    while True:
        run(n % w.h_q)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 8:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * f_one / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(),
            "kind": "oracle",
            "sample": f"{n} query head(s) of sequence 0, length {L}, fp64 numpy oracle, "
                      f"{dt:.1f} s"}


def run_reference(args, budget_s=120.0):
    """The oracle on the host cores, each step the same bounded slice of the
    workload (one query head's last n query rows), n sized from one timed
    calibration call so that the warm-up and timed steps take about
    ``budget_s`` together."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    x = synth.make_inputs(w)
    L = x.lengths[0] if w.varlen else w.seqlen_q
    n0 = min(L, 256)
    run0, _, _, _ = oracle_sample(w, x, n0)
    t0 = time.perf_counter()
    run0(0)
    per_row = (time.perf_counter() - t0) / n0
    want = budget_s / (args.steps + args.warmup) / max(per_row, 1e-9)
    n = L if want >= L else max(64, int(want) // 64 * 64)
    run, f_one, L, n = oracle_sample(w, x, n)
    for i in range(args.warmup):
        run(i % w.h_q)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        run(i % w.h_q)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    val = f_one / (ms * 1e-3) / 1e12
    sample = (f"one query head of sequence 0 per step: its last {n} of {L} query rows against "
              f"every key they see, fp64 numpy oracle")
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), seeded",
           "config": {"workload": w.name, "sample": sample},
           "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": _cores(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--pass", dest="pass_", default="bwd", choices=["bwd", "fwd"],
                    help="bwd: the backward (default); fwd: the forward that makes O and LSE")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--chunks", type=int, default=0,
                    help="attn_bwd_host chunk count for the end-to-end number (0: library default)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
    elif args.pass_ == "fwd":
        run_ours_fwd(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
