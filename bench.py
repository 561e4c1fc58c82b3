"""Benchmark: SageAttention3 NVFP4 attention forward on GB300.

One step = the whole hot path over one batch: quantize Q, K, V (bf16 -> NVFP4)
and the fused FP4 attention forward.  Metric: TOPS = 4*B*H*N^2*D / t (causal
counted at half).  Inputs are synthetic and seeded (bit_attention_gb300.synth);
the default workload is B4 H32 N4096 D128 (LLM-prefill shape with K outlier
channels), whose bf16 inputs (384 MiB) exceed L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle timed on the host cores

Prints one JSON line (rank 0).  Under torchrun the ranks split one problem's
B*H heads between them (--partition heads, the default: strong scaling, no
data-path collective), or each rank runs its own batch of the workload
(--partition batch: weak scaling).  With one GPU the line also carries a
per_workload block: the same kernels timed on every benchmark workload, and
a sagebwd block: the 8-bit training attention (forward + backward) on its
two training shapes.

  python bench.py --path sagebwd [--workload train_llama1b|train_qwen3b]

times SageBwd alone: one step = quantize Q, K, V, the forward, the backward
preparation (dO), the backward (dK, dV, dQ) and dQ's output, on the seeded
synthetic training inputs; metric TOPS = 3.5 * 4*B*H*N^2*D / t (the
backward's five products counted as 2.5 forwards; causal at half).
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

METRIC = "NVFP4 attention fwd TOPS (4*B*H*N^2*D/t) on 1 GB300; % of dense FP4 peak"
FP4_OVER_BF16 = 6.0  # nominal dense FP4 / BF16 tensor rate (13.5 / 2.25 PFLOP/s)
# NVIDIA's published dense NVFP4 rate of one Blackwell Ultra (GB300) GPU, an
# external figure reported beside the measured denominators
FP4_PUBLISHED_TFLOPS = 15000.0
HBM_NOMINAL_GBS = 8000.0  # the "~8 TB/s" HBM3e figure the quantize target is quoted against


TRAIN_METRIC = ("SageBwd 8-bit attention fwd+bwd TOPS (3.5*4*B*H*N^2*D/t, causal at half) on 1 GB300; "
                "fraction of the measured dense 16-bit tensor peak (tcgen05 kind::f16)")
SAGEBWD_CALLS = ("quantize_qkv", "attn_fwd", "bwd_prep", "attn_bwd", "dq_out")

# dram__bytes_read.sum + dram__bytes_write.sum of one attn_fwd_kernel launch,
# captured with ncu on this build of the kernel, mean of two launches (reads
# 113.32 MB = the compulsory Q, K, V codes and scales; writes 80.14 MB of the
# 134.2 MB O, the rest leaves L2 after the launch).  Workloads without a capture report null.
ATTN_TRAFFIC = {
    "attn_fwd B4 H32 N4096 D128 k-channel-outliers": 113.32e6 + 80.14e6,
}
# the same for one SageBwd attn_bwd launch (dkdv_tc_kernel).  The last ncu
# capture (B1 H16 N8192 D64 causal: 118.59 MB read, 28.40 MB written; B1 H8
# N8192 D128 causal: 184.29 MB read, 43.82 MB written) predates the change of
# the kernel's CTA dispatch order, which can move L2 reuse, so no figure is
# claimed for the current kernel: null until it is captured again.
SAGEBWD_BWD_TRAFFIC = {}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "hbm_gbs": p["hbm_gbs"], "src": "measured"}
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        loaded = [x for x in sm if mx and x > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: the job finishes when every rank has."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ops_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job TOPS: every rank processes its own batch (weak scaling)."""
    return ops_per_rank * world / (ms_per_step_max * 1e-3) / 1e12


def problem_throughput(ops_total: float, ms_per_step_max: float) -> float:
    """Whole-job TOPS when the ranks split one problem (strong scaling): the
    problem's work over the slowest rank's time."""
    return ops_total / (ms_per_step_max * 1e-3) / 1e12


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_sample(w, target_s: float, seed: int = 0, fmt: str = "nvfp4"):
    """Time the oracle's path (quantization + attention) on a bounded row
    sample of workload w: one (b,h) with the full N, Q, K and V quantized in
    full, then attention on random query rows until about target_s seconds
    of attention have run.  The quantization time is charged pro rata, the
    sampled rows' share of the head's N rows.  Returns (TOPS, seconds, rows,
    threads, quantize seconds of the whole head)."""
    import numpy as np
    import oracle
    from bit_attention_gb300.synth import make_qkv
    # a reduced batch with the same per-row work (full N, same D and pattern)
    q, k, v = make_qkv(1, 1, w.N, w.D, w.pattern, seed=seed)
    lnorm = "rounded" if fmt == "mxfp4_directp" else "exp"  # Direct-P: MXFP4, rounded normaliser
    t0 = time.perf_counter()
    qz = oracle.Quantized(q, k, v, 1, w.N, w.D, fmt="mxfp4" if fmt == "mxfp4_directp" else fmt)
    quant_s = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    rows_done, secs, ops = 0, 0.0, 0.0
    batch = max(oracle.num_threads(), 1)
    while secs < target_s:
        rows = rng.integers(0, w.N, size=batch)
        t0 = time.perf_counter()
        oracle.attention(qz, w.causal, rows=rows, lnorm=lnorm)
        secs += time.perf_counter() - t0
        keys = (rows + 1) if w.causal else np.full(batch, w.N)
        ops += float((4.0 * keys * w.D).sum())
        rows_done += batch
        batch = min(batch * 2, 1024)
    secs += quant_s * rows_done / w.N
    return ops / secs / 1e12, secs, rows_done, oracle.num_threads(), quant_s


def run_reference(args, w, world, rank):
    """--impl reference: the CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    tops = []
    rows_total, threads = 0, 1
    for i in range(args.warmup + args.steps):
        v, secs, rows, threads, _ = cpu_oracle_sample(w, args.ref_seconds, seed=i, fmt=args.fmt)
        if i >= args.warmup:
            tops.append(v)
            rows_total += rows
    value = statistics.mean(tops)
    sample = (f"oracle path (FP64 C, OpenMP) per step: Q, K, V of one (b,h) of the workload "
              f"quantized in full (N={w.N}, charged pro rata to the sampled rows), attention on "
              f"~{rows_total // max(args.steps, 1)} random query rows of it; ms_per_step "
              f"extrapolated: the whole workload at the sampled rate")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
           "ms_per_step": w.ops / (value * 1e12) * 1e3 if value > 0 else None,
           "extrapolated": True, "extrapolated_fields": ["ms_per_step"],
           "dtype": "f64", "data": "synthetic",
           "config": dict(w.describe(), format=args.fmt),
           "cpu_baseline": {"value": value, "unit": "TOPS", "cores": threads, "kind": "oracle",
                            "sample": sample, "extrapolated": True},
           "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def time_path(S, w, qd, kd, vd, z, o, fmt, steps, warmup, stream):
    """Warm up, then time `steps` steps (quantize + attention) with CUDA
    events on `stream`.  Returns (total ms, per-step quantize ms, per-step
    attention ms)."""
    import torch

    for _ in range(warmup):
        S.quantize_qkv(qd, kd, vd, out=z, fmt=fmt)
        S.attn_fwd(z, w.causal, out=o)
    torch.cuda.synchronize()
    if z.get_status() != 0:
        raise RuntimeError("kernel status nonzero after warm-up")
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        S.quantize_qkv(qd, kd, vd, out=z, fmt=fmt)
        e1.record(stream)
        S.attn_fwd(z, w.causal, out=o)
        e2.record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    status = z.get_status()
    if status != 0:
        raise RuntimeError(f"kernel status {S.strerror(status)}")
    return (start.elapsed_time(end), [a.elapsed_time(b) for a, b, _ in ev],
            [b.elapsed_time(c) for _, b, c in ev])


def quant_bytes(w) -> int:
    """Algorithmic bytes of quantizing Q, K, V: 2 B read and 0.5 + 1/16 B written per element."""
    elems = w.B * w.H * w.N * w.D
    return 3 * elems * 2 + 3 * (elems // 2 + elems // 16)


def per_workload(S, names, fmt, steps, warmup, dev, stream, fp4_peak, hbm_gbs):
    """The same kernels timed on each named workload (fewer steps than the
    headline); inputs are the seeded synthetic ones of that workload."""
    import torch
    from bit_attention_gb300.synth import WORKLOADS, make_workload
    out = {}
    for name in names:
        w = WORKLOADS[name]
        q, k, v = make_workload(w, seed=0)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        del q, k, v
        z = S.QuantizedQKV(w.B, w.H, w.N, w.D, device=dev)
        o = torch.empty_like(qd)
        _, q_ms, a_ms = time_path(S, w, qd, kd, vd, z, o, fmt, steps, warmup, stream)
        am, qm = statistics.mean(a_ms), statistics.mean(q_ms)
        tops = w.ops / (am * 1e-3) / 1e12
        gbs = quant_bytes(w) / (qm * 1e-3) / 1e9
        out[name] = {"workload": w.name, "steps": steps, "attn_ms": am, "attn_tops": tops,
                     "attn_frac_of_fp4_peak": tops / fp4_peak,
                     "attn_frac_of_fp4_published": tops / FP4_PUBLISHED_TFLOPS,
                     "quant_ms": qm, "quant_gbs": gbs, "quant_frac_of_hbm_measured": gbs / hbm_gbs,
                     "quant_frac_of_hbm_8tbs": gbs / HBM_NOMINAL_GBS,
                     "step_tops": w.ops / ((am + qm) * 1e-3) / 1e12}
        del qd, kd, vd, z, o
        torch.cuda.empty_cache()
    return out


class SageBwdRun:
    """Device buffers of one SageBwd training step on workload w, and its
    five C-ABI step calls on `stream`."""

    def __init__(self, SB, w, dev, seed=0):
        import torch
        from bit_attention_gb300.synth import make_dout, make_qkv
        self.SB, self.w = SB, w
        q, k, v = make_qkv(w.B, w.H, w.N, w.D, w.pattern, seed)
        do = make_dout(w.B, w.H, w.N, w.D, seed)
        self.host = (q, k, v, do)
        self.q, self.k, self.v, self.do = (t.to(dev) for t in self.host)
        self.ws = SB.Workspace(w.B, w.H, w.N, w.D, dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.scale = w.D ** -0.5

    def calls(self, stream):
        SB, w, ws = self.SB, self.w, self.ws
        dims = (w.B, w.H, w.N, w.D)
        wsa = (ws.buf.data_ptr(), ws.nbytes, stream.cuda_stream)
        c, sc = int(w.causal), self.scale
        p = lambda t: t.data_ptr()
        return (
            lambda: SB.sagebwd_quantize_qkv(p(self.q), p(self.k), p(self.v), *dims, *wsa),
            lambda: SB.sagebwd_attn_fwd(p(self.o), p(self.lse), *dims, c, sc, *wsa),
            lambda: SB.sagebwd_bwd_prep(p(self.do), p(self.o), p(self.lse), *dims, *wsa),
            lambda: SB.sagebwd_attn_bwd(p(self.dk), p(self.dv), *dims, c, sc, *wsa),
            lambda: SB.sagebwd_dq_out(p(self.dq), *dims, *wsa),
        )

    def time(self, steps, warmup, stream):
        """Time `steps` steps, each of the five calls between CUDA events.
        Returns (total ms, {call: [ms per step]})."""
        import torch
        calls = self.calls(stream)
        for _ in range(warmup):
            for fn in calls:
                if fn() != 0:
                    raise RuntimeError("SageBwd call failed")
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
        for i in range(steps):
            ev[i][0].record(stream)
            for j, fn in enumerate(calls):
                fn()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        status = self.ws.get_status(stream)
        if status != 0:
            raise RuntimeError(f"SageBwd kernel status {status}")
        per = {nm: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]
               for j, nm in enumerate(SAGEBWD_CALLS)}
        return ev[0][0].elapsed_time(ev[-1][-1]), per


def sagebwd_peak():
    """The tensor peak the SageBwd attention kernels are judged against: they
    issue tcgen05.mma kind::f16, so the measured dense 16-bit GEMM peak (FP16
    and BF16 share the nominal rate)."""
    pk = peaks()
    return pk["bf16_tflops"], f"{pk['src']} bf16 GEMM (burst), the tcgen05 kind::f16 rate"


def sagebwd_summary(w, per):
    """Per-call means and the roofline figures of the two attention kernels."""
    m = {nm: statistics.mean(v) for nm, v in per.items()}
    ops = w.ops
    fwd_tops = ops / (m["attn_fwd"] * 1e-3) / 1e12
    bwd_tops = 2.5 * ops / (m["attn_bwd"] * 1e-3) / 1e12
    step = sum(m.values())
    peak, src = sagebwd_peak()
    return {"workload": w.name, "ms": m, "ms_per_step": step,
            "attn_fwd_tops": fwd_tops, "attn_bwd_tops": bwd_tops,
            "peak_tflops": peak, "peak_src": src,
            "attn_fwd_frac_of_peak": fwd_tops / peak,
            "attn_bwd_frac_of_peak": bwd_tops / peak,
            "step_tops": 3.5 * ops / (step * 1e-3) / 1e12}


def sagebwd_cpu_sample(w, seed=0):
    """The SageBwd oracle (FP64 C, OpenMP) on one head of workload w at its
    full N: forward and backward.  Returns (TOPS, seconds, threads)."""
    import oracle
    from bit_attention_gb300.synth import make_dout, make_qkv
    q, k, v = make_qkv(1, 1, w.N, w.D, w.pattern, seed)
    do = make_dout(1, 1, w.N, w.D, seed)
    t0 = time.perf_counter()
    oracle.sagebwd(q, k, v, do, 1, w.N, w.D, w.causal)
    secs = time.perf_counter() - t0
    head_ops = 3.5 * w.ops / (w.B * w.H)
    return head_ops / secs / 1e12, secs, oracle.num_threads()


def run_sagebwd(args, world, rank, local):
    """--path sagebwd: the SageBwd training step alone (one GPU; under
    torchrun every rank runs its own batch: weak scaling)."""
    from bit_attention_gb300.synth import TRAIN_WORKLOADS
    w = TRAIN_WORKLOADS[args.workload if args.workload in TRAIN_WORKLOADS else "train_llama1b"]
    if args.impl == "reference":
        if rank != 0:
            return
        vals, secs_all, threads = [], [], 1
        for i in range(args.warmup + args.steps):
            v, secs, threads = sagebwd_cpu_sample(w, seed=i)
            if i >= args.warmup:
                vals.append(v)
                secs_all.append(secs)
        value = statistics.mean(vals)
        sample = (f"SageBwd oracle (FP64 C, OpenMP) per step: forward and backward of one (b,h) of the "
                  f"workload at full N={w.N} ({statistics.mean(secs_all):.1f} s); ms_per_step "
                  f"extrapolated: the whole workload at that rate")
        print(json.dumps({
            "impl": "reference", "metric": TRAIN_METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "ms_per_step": 3.5 * w.ops / (value * 1e12) * 1e3, "extrapolated": True,
            "extrapolated_fields": ["ms_per_step"], "dtype": "f64", "data": "synthetic",
            "config": w.describe(),
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": threads, "kind": "oracle",
                             "sample": sample, "extrapolated": True},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return

    import torch
    from bit_attention_gb300 import sagebwd as SB
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    run = SageBwdRun(SB, w, dev, seed=rank)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, per = run.time(args.steps, args.warmup, stream)
    barrier(world)
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    value = job_throughput(3.5 * w.ops, world, ms_step)
    summ = sagebwd_summary(w, per)

    # end to end through the public API with host buffers: every step copies
    # q, k, v, dout from pinned host memory, runs forward and backward, and
    # copies o, dq, dk, dv back
    e2e = None
    if not args.no_e2e:
        hin = [t.pin_memory() for t in run.host]
        hout = [torch.empty(run.o.shape, dtype=run.o.dtype, pin_memory=True) for _ in range(4)]
        calls = run.calls(stream)
        dins = (run.q, run.k, run.v, run.do)
        douts = (run.o, run.dq, run.dk, run.dv)

        def e2e_step():
            for d, h in zip(dins, hin):
                d.copy_(h, non_blocking=True)
            for fn in calls:
                fn()
            for h, d in zip(hout, douts):
                h.copy_(d, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(s0.elapsed_time(s1), world) / args.steps
        elems = w.B * w.H * w.N * w.D
        e2e = {"value": job_throughput(3.5 * w.ops, world, e2e_ms), "unit": "TOPS", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": 4 * elems * 2, "d2h_bytes_per_step": 4 * elems * 2,
               "call": "sagebwd_quantize_qkv, _attn_fwd, _bwd_prep, _attn_bwd, _dq_out with pinned-host copies"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v_cpu, secs, threads = sagebwd_cpu_sample(w)
        cpu = {"value": v_cpu, "unit": "TOPS", "cores": threads, "kind": "oracle", "extrapolated": False,
               "sample": f"SageBwd oracle: forward and backward of one (b,h) of the workload at full N={w.N}, "
                         f"{secs:.1f} s; the value is the rate on that head"}
    if rank == 0:
        print(json.dumps({
            "metric": TRAIN_METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8 codes (per-block scales) on the fp16 tensor path, exact integer sums / fp16 dP / "
                     "fp32 accumulate",
            "data": "synthetic (seeded, bit_attention_gb300.synth)",
            "config": dict(w.describe(), l2="bf16 inputs 4x32 MiB+ per tensor set; no flush",
                           parallelism=f"weak, {world} independent batch(es)"),
            "kernels": summ,
            "roofline": {"bound": "tensor",
                         "kernel": "attn_bwd (dkdv_tc_kernel)",
                         "achieved": summ["attn_bwd_tops"], "peak": summ["peak_tflops"], "unit": "TFLOP/s",
                         "frac": summ["attn_bwd_frac_of_peak"], "traffic": SAGEBWD_BWD_TRAFFIC.get(w.name),
                         "traffic_unit": "DRAM bytes (read + write) per attn_bwd launch, from ncu",
                         "peak_src": summ["peak_src"]},
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk.summary(),
            "gpu_launches": len(SAGEBWD_CALLS) * args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llm")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--causal", type=int, default=None)
    ap.add_argument("--shape", default=None, help="B,H,N,D override (profiling cases)")
    ap.add_argument("--fmt", default="nvfp4", choices=["nvfp4", "mxfp4", "mxfp4_directp"],
                    help="microscaling format (mxfp4: the variant the pages set aside; "
                         "mxfp4_directp: MXFP4 with the normaliser from the rounded P)")
    ap.add_argument("--partition", default="heads", choices=["heads", "batch"],
                    help="with several ranks: split one problem's heads (strong scaling) or run "
                         "one batch per rank (weak scaling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sdpa", action="store_true", help="skip the bf16 SDPA context timing")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload block (one GPU only)")
    ap.add_argument("--path", default="fp4", choices=["fp4", "sagebwd"],
                    help="fp4: the NVFP4 inference attention (the headline); sagebwd: the 8-bit "
                         "training attention, forward + backward")
    ap.add_argument("--no-sagebwd", action="store_true", help="skip the sagebwd block (one GPU only)")
    ap.add_argument("--ref-seconds", type=float, default=6.0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    if args.path == "sagebwd":
        world, rank, local = dist_init()
        run_sagebwd(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    from bit_attention_gb300.synth import WORKLOADS, Workload
    w = WORKLOADS[args.workload]
    if args.causal is not None:
        w = Workload(w.name, w.B, w.H, w.N, w.D, bool(args.causal), w.pattern)
    if args.shape:
        B, H, N, D = (int(x) for x in args.shape.split(","))
        w = Workload(f"attn_fwd B{B} H{H} N{N} D{D} {w.pattern}", B, H, N, D, w.causal, w.pattern)

    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return

    import torch
    from bit_attention_gb300 import sage_fp4 as S
    from bit_attention_gb300.shard import head_view, shard_heads
    from bit_attention_gb300.synth import make_workload
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    strong = world > 1 and args.partition == "heads"
    if strong:
        # every rank draws the same problem and keeps its share of the heads
        q, k, v = make_workload(w, seed=0)
        first, count = shard_heads(w.B, w.H, rank, world)
        q, k, v = (head_view(t, first, count).contiguous() for t in (q, k, v))
        wr = Workload(w.name, 1, count, w.N, w.D, w.causal, w.pattern)
    else:
        q, k, v = make_workload(w, seed=rank)
        wr = w
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    z = S.QuantizedQKV(wr.B, wr.H, wr.N, wr.D, device=dev)
    o = torch.empty_like(qd)
    stream = torch.cuda.current_stream()

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, q_all, a_all = time_path(S, wr, qd, kd, vd, z, o, args.fmt, args.steps,
                                           args.warmup, stream)
    barrier(world)
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    q_ms = statistics.mean(q_all)
    a_ms = statistics.mean(a_all)

    ops = wr.ops  # this rank's work per step
    value = problem_throughput(w.ops, ms_step) if strong else job_throughput(ops, world, ms_step)
    pk = peaks()
    fp4_peak = pk["bf16_tflops"] * FP4_OVER_BF16
    attn_tops = ops / (a_ms * 1e-3) / 1e12
    elems = wr.B * wr.H * wr.N * wr.D
    quant_gbs = quant_bytes(wr) / (q_ms * 1e-3) / 1e9

    # end to end through the public API: one C-ABI call with pinned host
    # buffers per step (sage_fp4_attention_host: host -> device copies,
    # quantize, attention and the copy of O back to host memory, pipelined
    # over chunks of heads inside the library)
    e2e = None
    if not args.no_e2e and args.fmt == "nvfp4":
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hws = S.HostWorkspace(wr.B, wr.H, wr.N, wr.D)

        def e2e_step():
            S.attention_host(hq, hk, hv, wr.causal, out=ho, workspace=hws, stream=stream)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(s0.elapsed_time(s1), world) / args.steps
        e2e_value = (problem_throughput(w.ops, e2e_ms) if strong
                     else job_throughput(ops, world, e2e_ms))
        e2e = {"value": e2e_value, "unit": "TOPS",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * elems * 2,
               "d2h_bytes_per_step": elems * 2, "call": "sage_fp4_attention_host",
               "head_chunks": -(-(wr.B * wr.H) // -(-(wr.B * wr.H) // 8))}

    # context only (not a target): PyTorch's bf16 scaled_dot_product_attention
    # on the same inputs and GPU, outside the timed region
    context = None
    if not args.no_sdpa:
        try:
            import torch.nn.functional as F
            for _ in range(2):
                F.scaled_dot_product_attention(qd, kd, vd, is_causal=wr.causal)
            torch.cuda.synchronize()
            times = []
            for _ in range(5):
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
                F.scaled_dot_product_attention(qd, kd, vd, is_causal=wr.causal)
                s1.record(stream)
                torch.cuda.synchronize()
                times.append(s0.elapsed_time(s1))
            sdpa_ms = statistics.median(times)
            context = {"sdpa_bf16_ms": sdpa_ms, "sdpa_bf16_tops": ops / (sdpa_ms * 1e-3) / 1e12,
                       "attn_kernel_speedup_vs_sdpa_bf16": sdpa_ms / a_ms}
        except Exception as exc:  # context only
            context = {"sdpa_bf16": f"unavailable: {type(exc).__name__}"}

    # context: the rate the tensor cores sustain on the attention kernel's own
    # MMA instruction (back-to-back, operands in shared memory), after the
    # timed region
    fp4_mma = S.mma_peak_tflops(n=256)

    # the same kernels on every benchmark workload (one GPU only; fewer steps)
    pw = None
    if world == 1 and not args.no_per_workload and args.shape is None and args.causal is None:
        del qd, kd, vd, z, o
        torch.cuda.empty_cache()
        names = [n for n in ("llm", "llm_causal", "dit", "dit_long") if n != args.workload]
        pw = per_workload(S, names, args.fmt, steps=5, warmup=3, dev=dev, stream=stream,
                          fp4_peak=fp4_peak, hbm_gbs=pk["hbm_gbs"])
        pw[args.workload] = {"workload": wr.name, "steps": args.steps, "attn_ms": a_ms,
                             "attn_tops": attn_tops, "attn_frac_of_fp4_peak": attn_tops / fp4_peak,
                             "attn_frac_of_fp4_published": attn_tops / FP4_PUBLISHED_TFLOPS,
                             "quant_ms": q_ms, "quant_gbs": quant_gbs,
                             "quant_frac_of_hbm_measured": quant_gbs / pk["hbm_gbs"],
                             "quant_frac_of_hbm_8tbs": quant_gbs / HBM_NOMINAL_GBS,
                             "step_tops": ops / ((a_ms + q_ms) * 1e-3) / 1e12, "headline": True}

    # the 8-bit training attention on its two training shapes (one GPU only)
    sbw = None
    if world == 1 and not args.no_sagebwd and args.shape is None and args.causal is None:
        from bit_attention_gb300 import sagebwd as SB
        from bit_attention_gb300.synth import TRAIN_WORKLOADS
        torch.cuda.empty_cache()
        sbw = {"metric": TRAIN_METRIC}
        for name in ("train_llama1b", "train_qwen3b"):
            run = SageBwdRun(SB, TRAIN_WORKLOADS[name], dev)
            _, per = run.time(5, 3, stream)
            sbw[name] = sagebwd_summary(run.w, per)
            del run
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v_cpu, secs, rows, threads, quant_s = cpu_oracle_sample(w, args.cpu_seconds, fmt=args.fmt)
        cpu = {"value": v_cpu, "unit": "TOPS", "cores": threads, "kind": "oracle",
               "extrapolated": False,
               "sample": f"oracle path on one (b,h) of the workload, full N={w.N}: Q, K, V "
                         f"quantized in full ({quant_s:.2f} s, charged pro rata) and attention on "
                         f"{rows} random query rows; {secs:.1f} s in all; the value is the rate on "
                         f"that sample"}

    if rank == 0:
        par = (f"heads: one problem's {w.B * w.H} heads split over {world} ranks" if strong
               else f"weak, {world} independent batch(es)")
        out = {
            "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "strong" if strong else "weak",
            "vs_baseline": None,
            "dtype": ("nvfp4 (e2m1 codes, e4m3 scales)" if args.fmt == "nvfp4"
                      else "mxfp4 (e2m1 codes, e8m0 scales)") + " / fp32 accumulate" +
                     (", normaliser from the rounded P (Direct-P)" if args.fmt == "mxfp4_directp" else ""),
            "data": "synthetic (seeded, bit_attention_gb300.synth)",
            "config": dict(w.describe(), format=args.fmt, l2="bf16 inputs 3x larger than L2; no flush",
                           parallelism=par),
            "attn_kernel": {"ms": a_ms, "tops": attn_tops, "frac_of_fp4_peak": attn_tops / fp4_peak,
                            "ms_median": statistics.median(a_all), "ms_min": min(a_all),
                            "ms_max": max(a_all)},
            "context": context,
            "quant_kernels": {"ms": q_ms, "gbs": quant_gbs,
                              "frac_of_hbm": quant_gbs / pk["hbm_gbs"],
                              "frac_of_hbm_8tbs": quant_gbs / HBM_NOMINAL_GBS},
            "roofline": {"bound": "tensor", "achieved": attn_tops, "peak": fp4_peak,
                         "unit": "TFLOP/s", "frac": attn_tops / fp4_peak,
                         "traffic": ATTN_TRAFFIC.get(wr.name) if args.fmt == "nvfp4" else None,
                         "traffic_unit": "DRAM bytes (read + write) per attention launch, from ncu",
                         "peak_src": f"{pk['src']} bf16 x {FP4_OVER_BF16:g} (nominal FP4/BF16)",
                         "peak_published_tflops": FP4_PUBLISHED_TFLOPS,
                         "frac_of_published": attn_tops / FP4_PUBLISHED_TFLOPS,
                         "fp4_mma_measured_tflops": fp4_mma,
                         "frac_of_fp4_mma_measured": attn_tops / fp4_mma},
            "per_workload": pw, "sagebwd": sbw,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clk.summary(),
            "gpu_launches": 3 * args.steps,
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
