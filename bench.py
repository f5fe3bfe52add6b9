"""Benchmark: fused attention + Ulysses All-to-All layout on GB300.

One step = one call of the fused path (attention over [B,S,H,D] with every
output tile stored into its owner's sequence shard) on one batch of seeded
synthetic bf16 input already resident in HBM.  Metric: TFLOP/s of the
4*B*H*S^2*D tensor FLOPs, whole-job (summed over ranks).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload video_large]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

Prints ONE JSON line (rank 0).  Between timed steps the L2 cache is flushed by
writing a 256 MiB buffer outside the timed events; each step is timed with CUDA
events on the launching stream and the per-step times are summed.
"""
from __future__ import annotations

import argparse
import hashlib
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

import numpy as np  # noqa: E402

import dit_inputs as di  # noqa: E402

DEFAULT_WORKLOAD = "video_large"
SIDE_WORKLOAD = "image"   # timed as an extra key of the default line
D64_WORKLOAD = "video_small_d64"   # the head-dimension-64 kernel, another extra key
METRIC = "fused attn+A2A-layout TFLOP/s and % of GB300 dense BF16 peak; fused-store overhead %"
KERNEL_SOURCES = ["dit_attention_ulysses_gb300/csrc/attn_fwd.cu", "dit_attention_ulysses_gb300/csrc/ptx.cuh",
                  "dit_attention_ulysses_gb300/csrc/kernels.h"]
PROFILES = os.path.join(ROOT, "profiles")


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def _read_summary(path):
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    return vals


# ex2.approx.ftz.f32 retired per SM clock per SM on GB300 with two warps per
# sub-partition (a probe issuing independent ex2 back to back measured 4.12 cycles
# per warp instruction per sub-partition: 4 x 32 / 4.12 = 31.1).
MUFU_EX2_PER_CLK_SM = 31.1


def mufu_bound(w, sm_mhz, sms):
    """The attainable rate if the B*H*S^2 exponentials (one per score, 4*D tensor
    FLOPs each) were the only limit, at the SM clock seen in the timed region."""
    if not sm_mhz:
        return None
    per_s = MUFU_EX2_PER_CLK_SM * sms * sm_mhz * 1e6
    return {"ex2_per_clk_per_sm": MUFU_EX2_PER_CLK_SM, "sm_mhz": sm_mhz,
            "bound_tflops": per_s * 4 * w.D / 1e12, "exps_per_step": w.B * w.H * w.S * w.S}


def tiles_of(w) -> int:
    return w.B * w.H * ((w.S + 127) // 128)


def ncu_traffic(w):
    """DRAM bytes per launch of the fused kernel from a committed ncu summary taken on
    the current kernel source: the workload's own capture, else a capture of a smaller
    workload scaled by query tiles (K/V of the head being worked on stay in L2, so every
    tile moves the same bytes: its Q and O tiles and its share of the head's K and V).
    Returns (bytes or None, note)."""
    names = sorted(f for f in os.listdir(PROFILES) if f.startswith("ncu_attn_a2a_kernel_") and f.endswith(".txt"))
    own = f"ncu_attn_a2a_kernel_{w.name}.txt"
    if own in names:
        names.remove(own)
        names.insert(0, own)
    for name in names:
        vals = _read_summary(os.path.join(PROFILES, name))
        if vals.get("kernel_source_sha256_16") != kernel_source_hash() or vals.get("head_dim", "128") != str(w.D):
            continue
        try:
            if vals.get("workload") == w.name:
                return int(float(vals["dram_bytes_per_launch_full_workload"])), f"ncu capture of {w.name} ({name})"
            per_tile = float(vals["dram_bytes_per_tile"])
        except (KeyError, ValueError):
            continue
        return int(per_tile * tiles_of(w)), (f"ncu capture of {vals.get('workload')} ({name}), "
                                             f"{per_tile:.0f} B per query tile x {tiles_of(w)} tiles")
    return None, "no ncu capture of the current kernel source"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 - 0.06 <= ts <= t1 + 0.06] or [r for _, r in rows[-3:]]
        sm = [float(r[0]) for r in inside if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host float over all ranks (gloo); identity for one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, ms_per_step: float, world: int) -> float:
    """Weak scaling: every rank processes its own copy of the workload."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def to_device(bits, torch, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def time_steps(torch, fn, steps, flush, stream, host_ms=None):
    """Run `steps` timed calls of fn with an L2 flush before each; returns per-step ms list.
    `host_ms`, when given, receives the host time each call took to return (enqueue)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.add_(1)
        starts[i].record(stream)
        t0 = time.perf_counter()
        fn()
        if host_ms is not None:
            host_ms.append((time.perf_counter() - t0) * 1e3)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def cpu_oracle_sample(w, seconds_target=12.0, max_rows=None, inputs=None):
    """Time the fp64 oracle on a bounded sample of query rows (all heads) of workload w.
    Returns the cpu_baseline object and (rows_b, rows_s, oracle rows [n, H, D])."""
    import oracle
    q, k, v = di.random_qkv(w) if inputs is None else inputs
    threads = oracle.threads_used()
    per_pair = 4.0 * w.S * w.D  # flops per (row, head)
    # calibrate on a sample large enough to occupy every thread for a while
    # (at least ~1 s), then size the timed sample for ~seconds_target
    n_cal, dt = 8 * threads, 0.0
    while True:
        rb, rs = di.sample_rows(w, n_cal, seed=5)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.scale, rb, rs)
        dt = time.perf_counter() - t0
        if dt >= 1.0 or len(rb) >= w.B * w.S:
            break
        n_cal *= 4
    rate = len(rb) * w.H * per_pair / max(dt, 1e-4)
    n = int(seconds_target * rate / (w.H * per_pair))
    n = max(8, min(n, w.B * w.S if max_rows is None else max_rows))
    rb, rs = di.sample_rows(w, n, seed=6)
    t0 = time.perf_counter()
    ref = oracle.attention_rows(q, k, v, w.scale, rb, rs)
    dt = time.perf_counter() - t0
    flops = len(rb) * w.H * per_pair
    line = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rb)} query rows x {w.H} heads of the {w.name} workload ({flops:.3e} FLOPs, "
                      f"{dt:.1f} s, fp64 C/OpenMP)"}
    return line, (rb, rs, ref)


def sampled_parity(w, outs, rb, rs, ref):
    """The fused output at the oracle's sampled rows against the oracle: max-abs error,
    relative L2 error and how many elements exceed the flat 2e-2 bar."""
    Sl = w.S // w.P
    got = np.stack([outs[int(s) // Sl][int(b), int(s) % Sl].float().cpu().numpy() for b, s in zip(rb, rs)])
    err = np.abs(got.astype(np.float64) - ref)
    return {"rows": int(len(rb)), "elements": int(err.size), "max_abs": float(err.max()),
            "rel_l2": float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)),
            "n_above_2e-2": int((err > 2e-2).sum()), "max_abs_ref": float(np.abs(ref).max()),
            "against": "fp64 oracle rows of the cpu_baseline sample (all heads)"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    w = di.WORKLOADS[args.workload]
    q, k, v = di.random_qkv(w)
    threads = oracle.threads_used()
    rows_per_step = max(4, int(args.ref_rows))
    per_pair = 4.0 * w.S * w.D
    for i in range(args.warmup):
        rb, rs = di.sample_rows(w, rows_per_step, seed=100 + i)
        oracle.attention_rows(q, k, v, w.scale, rb, rs)
    total_flops, total_t, n_rows = 0.0, 0.0, 0
    for i in range(args.steps):
        rb, rs = di.sample_rows(w, rows_per_step, seed=1000 + i)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.scale, rb, rs)
        total_t += time.perf_counter() - t0
        total_flops += len(rb) * w.H * per_pair
        n_rows += len(rb)
    value = total_flops / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D, "P": w.P,
                   "sample": f"{rows_per_step} query rows x all heads per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} query rows x {w.H} heads over {args.steps} steps"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def step_percentiles(ms):
    """p10, p50 and p90 of per-step times (ms), for any number of steps >= 1."""
    p10, p50, p90 = np.percentile(np.asarray(ms, dtype=np.float64), [10, 50, 90])
    return {"p10": float(p10), "p50": float(p50), "p90": float(p90)}


def varlen_mix(total: int, seed: int = 12345):
    """Sequence lengths covering `total` tokens: drawn uniformly in [total/16, total/2)
    from a seeded generator until they cover it, the last one cut to fit."""
    rng = np.random.default_rng(seed)
    lens = []
    while sum(lens) < total:
        lens.append(int(rng.integers(max(1, total // 16), max(2, total // 2))))
    lens[-1] -= sum(lens) - total
    return lens


def side_workload_line(torch, xs, args, dev, stream, flush, name=SIDE_WORKLOAD):
    """The fused call on another workload (the image-DiT shape, the D = 64 kernel),
    timed like the main line (L2 flushed before each step), reported beside it."""
    w = di.WORKLOADS[name]
    q, k, v = (to_device(x, torch, dev) for x in di.random_qkv(w))
    outs = [torch.empty((w.B, w.S // w.P, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(w.P)]
    ws = xs.Workspace.for_shape(w.B, w.S, w.H, w.D, device=dev) if args.schedule == "balanced" else None
    fn = lambda: xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, outs, w.scale, ws, stream)
    for _ in range(3):
        fn()
    n = max(10, min(args.steps, 50))
    ms = time_steps(torch, fn, n, flush, stream)
    if xs.xs_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error in the side workload")
    tflops = w.flops / (statistics.mean(ms) * 1e-3) / 1e12
    peak = measured_peaks()[0]
    return {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D, "P": w.P, "steps": n,
            "ms_per_step": statistics.mean(ms), "tflops": tflops,
            "frac_of_bf16_burst": tflops / peak if peak else None,
            "step_ms_percentiles": step_percentiles(ms), "api": "xs_attn_fwd_balanced"}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import dit_attention_ulysses_gb300 as xs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = di.WORKLOADS[args.workload]
    B, S, H, D, P = w.B, w.S, w.H, w.D, w.P
    qb, kb, vb = di.random_qkv(w)
    q, k, v = (to_device(x, torch, dev) for x in (qb, kb, vb))
    shard_shape = (B, S // P, H, D)
    outs = [torch.empty(shard_shape, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    contig = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    heads = [torch.empty((B, S, H // P, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    serial = [torch.empty(shard_shape, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # balanced schedule: the last partial wave of query tiles is spread over all
    # SMs through a workspace (None when the tiles fill whole waves)
    ws = xs.Workspace.for_shape(B, S, H, D, device=dev) if args.schedule == "balanced" else None

    def fused():
        xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, outs, w.scale, ws, stream)

    def alone():
        xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_CONTIGUOUS, [contig], w.scale, ws, stream)

    def serial_path():
        xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_HEADS, heads, w.scale, ws, stream)
        xs.xs_relayout_a2a(heads, serial, stream)

    # the whole Ulysses step with the inputs as P sequence shards (both exchanges
    # fused), and its unfused form: pre-attention re-layout of Q, K, V, attention of
    # each rank on its head shard, post-attention re-layout
    Sl, Hl = S // P, H // P
    uly = Sl % 128 == 0
    if uly:
        q_sh, k_sh, v_sh = ([X[:, p * Sl:(p + 1) * Sl].contiguous() for p in range(P)] for X in (q, k, v))
        uly_out = [torch.empty(shard_shape, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        pre = [[torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device=dev) for _ in range(P)] for _ in range(3)]
        o_heads = [torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]
        uly_serial = [torch.empty(shard_shape, dtype=torch.bfloat16, device=dev) for _ in range(P)]

        def ulysses_fused():
            xs.xs_attn_ulysses_fwd(q_sh, k_sh, v_sh, uly_out, w.scale, ws, stream)

        def ulysses_serial():
            for src, dst in zip((q_sh, k_sh, v_sh), pre):
                xs.xs_relayout_a2a_inverse(src, dst, stream)
            for r in range(P):
                xs.xs_attn_fwd(pre[0][r], pre[1][r], pre[2][r], o_heads[r], w.scale, stream)
            xs.xs_relayout_a2a(o_heads, uly_serial, stream)

    # causal variant (row s attends to keys 0 .. s) with the same fused A2A stores
    causal_out = [torch.empty(shard_shape, dtype=torch.bfloat16, device=dev) for _ in range(P)]

    def causal():
        xs.xs_attn_causal_fwd(q, k, v, xs.XS_LAYOUT_A2A, causal_out, w.scale, stream)

    # packed variable-length sequences: the same B*S tokens, bidirectional within each
    T = B * S
    seqlens = varlen_mix(T)
    q_p, k_p, v_p = (x.view(T, H, D) for x in (q, k, v))
    varlen_out = [torch.empty((T // P, H, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]

    def varlen():
        xs.xs_attn_varlen_fwd(q_p, k_p, v_p, seqlens, xs.XS_LAYOUT_A2A, varlen_out, w.scale, False, stream)

    def varlen_causal():   # one causal launch per sequence
        xs.xs_attn_varlen_fwd(q_p, k_p, v_p, seqlens, xs.XS_LAYOUT_A2A, varlen_out, w.scale, True, stream)

    for _ in range(max(3, args.warmup)):
        fused()
    torch.cuda.synchronize()
    if xs.xs_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error during warm-up")

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    per_step = time_steps(torch, fused, args.steps, flush, stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    status = xs.xs_attn_get_device_error(stream)
    if status != 0:
        raise RuntimeError(f"device error status {status}")

    total_ms = max_over_ranks(sum(per_step), world)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(w.flops, ms_per_step, world)

    # ablation: attention alone (contiguous store), fused, and attention + separate
    # re-layout, interleaved run by run so that clock drift affects all three alike
    n_abl = max(10, min(args.steps, 50))
    for fn in (alone, serial_path, causal, varlen, varlen_causal) + ((ulysses_fused, ulysses_serial) if uly else ()):
        for _ in range(3):
            fn()
    ta, tf, ts, tc, tv, tvc, tuf, tus = [], [], [], [], [], [], [], []
    for _ in range(n_abl):
        ta += time_steps(torch, alone, 1, flush, stream)
        tf += time_steps(torch, fused, 1, flush, stream)
        ts += time_steps(torch, serial_path, 1, flush, stream)
        tc += time_steps(torch, causal, 1, flush, stream)
        tv += time_steps(torch, varlen, 1, flush, stream)
        tvc += time_steps(torch, varlen_causal, 1, flush, stream)
        if uly:
            tuf += time_steps(torch, ulysses_fused, 1, flush, stream)
            tus += time_steps(torch, ulysses_serial, 1, flush, stream)
    t_alone, t_fused, t_serial = statistics.median(ta), statistics.median(tf), statistics.median(ts)
    # causal tensor FLOPs: 4*D per unmasked (query, key) pair, S*(S+1)/2 pairs per (b, h)
    causal_flops = 2 * B * H * D * S * (S + 1)
    t_causal = statistics.median(tc)
    causal_line = {"api": "xs_attn_causal_fwd", "ms": t_causal, "tflops": causal_flops / (t_causal * 1e-3) / 1e12,
                   "flops": causal_flops, "flops_rule": "4*B*H*D*S*(S+1)/2 (unmasked query-key pairs)",
                   "over_bidirectional_fused_ms": t_causal / t_fused, "runs": n_abl, "statistic": "median"}
    varlen_flops = 4 * H * D * sum(n * n for n in seqlens)
    t_varlen = statistics.median(tv)
    varlen_line = {"api": "xs_attn_varlen_fwd", "seqlens": seqlens, "ms": t_varlen,
                   "tflops": varlen_flops / (t_varlen * 1e-3) / 1e12, "flops": varlen_flops,
                   "flops_rule": "4*H*D*sum(len^2) (each sequence attends to itself)",
                   "runs": n_abl, "statistic": "median"}
    varlen_causal_flops = 2 * H * D * sum(n * (n + 1) for n in seqlens)
    t_varlen_causal = statistics.median(tvc)
    varlen_causal_line = {"api": "xs_attn_varlen_fwd(causal=1)", "ms": t_varlen_causal,
                          "tflops": varlen_causal_flops / (t_varlen_causal * 1e-3) / 1e12,
                          "flops": varlen_causal_flops,
                          "flops_rule": "4*H*D*sum(len*(len+1)/2) (unmasked query-key pairs)",
                          "launches_per_call": sum(1 for n in seqlens if n > 0),
                          "runs": n_abl, "statistic": "median"}
    ulysses = None
    if uly:
        t_uf, t_us = statistics.median(tuf), statistics.median(tus)
        ulysses = {"api": "xs_attn_ulysses_fwd", "fused_step_ms": t_uf, "fused_step_tflops": w.flops / (t_uf * 1e-3) / 1e12,
                   "unfused_step_ms": t_us, "unfused_over_fused": t_us / t_uf,
                   "fused_step_over_whole_tensor_fused": t_uf / t_fused,
                   "unfused": "pre-attention re-layout of Q, K, V + attention per rank + post-attention re-layout",
                   "runs": n_abl, "statistic": "median"}

    # end to end through the host-buffer entry point: H2D of q, k, v, kernel, D2H of the shards
    pin = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = pin(qb), pin(kb), pin(vb)
    out_h = [torch.empty(shard_shape, dtype=torch.bfloat16).pin_memory() for _ in range(P)]
    e2e_fn = lambda: xs.xs_attn_a2a_fwd_staged(qh, kh, vh, out_h, q, k, v, outs, w.scale, workspace=ws, stream=stream)
    for _ in range(2):
        e2e_fn()
    n_e2e = max(3, min(args.steps, 20))
    e2e_host = []
    e2e_steps = time_steps(torch, e2e_fn, n_e2e, flush, stream, host_ms=e2e_host)
    e2e_ms = max_over_ranks(statistics.mean(e2e_steps), world)
    if xs.xs_attn_get_device_error(stream) != 0:
        raise RuntimeError("device error after ablation / e2e runs")
    side = side_workload_line(torch, xs, args, dev, stream, flush) if args.workload != SIDE_WORKLOAD else None
    d64 = side_workload_line(torch, xs, args, dev, stream, flush, D64_WORKLOAD) if w.D != 64 else None

    if rank != 0:
        return
    peak_tflops, _, peak_kind = measured_peaks()
    traffic, traffic_note = ncu_traffic(w)
    achieved = w.flops / (statistics.mean(per_step) * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "step_ms_percentiles": step_percentiles(per_step),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": B, "S": S, "H": H, "D": D, "P": P, "scale": w.scale,
                   "inputs": "seeded bf16 N(0,1)" + (" with outlier channels" if w.outliers else ""),
                   "l2": "flushed between timed steps (256 MiB write outside the timed events)",
                   "schedule": args.schedule, "workspace_bytes": ws.nbytes if ws else 0,
                   "parallelism": f"{world} independent replica(s), one GPU each" if world > 1 else "1 GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops if peak_tflops else None,
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "traffic": traffic,
                     "traffic_source": traffic_note,
                     "algorithmic_bytes": 4 * w.tensor_bytes,
                     "mufu_bound": mufu_bound(w, (clocks or {}).get("sm_mhz"),
                                              torch.cuda.get_device_properties(dev).multi_processor_count)},
        "epilogue_store": {"bytes_per_step": w.tensor_bytes,
                           "gb_per_s": w.tensor_bytes / (ms_per_step * 1e-3) / 1e9,
                           "note": "output bytes stored by the fused epilogue over the step time"},
        "overhead_pct": 100.0 * (t_fused - t_alone) / t_alone,
        "ablation": {"attention_alone_ms": t_alone, "fused_ms": t_fused, "attention_plus_relayout_ms": t_serial,
                     "serial_over_fused": t_serial / t_fused, "runs": n_abl, "statistic": "median",
                     "order": "interleaved alone/fused/serial, L2 flushed before each"},
        "e2e": {"value": whole_job_tflops(w.flops, e2e_ms, world), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 3 * w.tensor_bytes, "d2h_bytes_per_step": w.tensor_bytes,
                "ms_per_step": e2e_ms, "step_ms_percentiles": step_percentiles(e2e_steps),
                "step_ms": [round(x, 2) for x in e2e_steps], "host_enqueue_ms": [round(x, 2) for x in e2e_host],
                "api": "xs_attn_a2a_fwd_staged"},
        "ulysses_step": ulysses,
        "causal": causal_line,
        "varlen": varlen_line,
        "varlen_causal": varlen_causal_line,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "kernel_source": kernel_source_hash(),
    }
    if side is not None:
        line["side_workload"] = side
    if d64 is not None:
        line["d64_workload"] = d64
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"], (rb, rs, ref) = cpu_oracle_sample(w, seconds_target=args.cpu_seconds,
                                                                inputs=(qb, kb, vb))
        line["sampled_parity"] = sampled_parity(w, outs, rb, rs, ref)
    line["wall_s_timed_region"] = t_wall1 - t_wall0
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """The sequence sweep (B=2, H=16, D=128, P=8, S = 1024 ... 131072 doubling): at
    each S the fused call, the same kernel storing contiguously (attention alone)
    and the same kernel into head shards followed by the separate re-layout kernel,
    interleaved run by run with L2 flushed before each; medians and p10/p90."""
    import torch

    import dit_attention_ulysses_gb300 as xs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    runs = max(20, args.steps)
    sampler = ClockSampler(0)
    sampler.start()
    t0 = time.time()
    points = []
    for S in di.SWEEP_S:
        w = di.sweep_workload(S)
        B, H, D, P = w.B, w.H, w.D, w.P
        q, k, v = (to_device(x, torch, dev) for x in di.random_qkv(w))
        outs = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]
        contig = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
        heads = [torch.empty((B, S, H // P, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]
        serial = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ws = xs.Workspace.for_shape(B, S, H, D, device=dev) if args.schedule == "balanced" else None
        fused = lambda: xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, outs, w.scale, ws, stream)
        alone = lambda: xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_CONTIGUOUS, [contig], w.scale, ws, stream)

        def serial_path():
            xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_HEADS, heads, w.scale, ws, stream)
            xs.xs_relayout_a2a(heads, serial, stream)

        for fn in (fused, alone, serial_path):
            for _ in range(3):
                fn()
        tf, ta, ts = [], [], []
        for _ in range(runs):
            tf += time_steps(torch, fused, 1, flush, stream)
            ta += time_steps(torch, alone, 1, flush, stream)
            ts += time_steps(torch, serial_path, 1, flush, stream)
        if xs.xs_attn_get_device_error(stream) != 0:
            raise RuntimeError(f"device error in the sweep at S={S}")
        mf, ma, ms_ = statistics.median(tf), statistics.median(ta), statistics.median(ts)
        points.append({"S": S, "flops": w.flops, "fused_ms": step_percentiles(tf), "alone_ms": step_percentiles(ta),
                       "alone_plus_relayout_ms": step_percentiles(ts),
                       "fused_tflops": w.flops / (mf * 1e-3) / 1e12,
                       "overhead_pct": 100.0 * (mf - ma) / ma, "serial_over_fused": ms_ / mf,
                       "schedule": "split" if ws is not None else "whole tiles"})
        del q, k, v, outs, contig, heads, serial, ws
        torch.cuda.empty_cache()
    clocks = sampler.stop(t0, time.time())
    peak_tflops, _, peak_kind = measured_peaks()
    for pt in points:
        pt["frac_of_peak"] = pt["fused_tflops"] / peak_tflops
    print(json.dumps({"sweep": points, "runs_per_point": runs, "statistic": "median (p10/p90 beside it)",
                      "order": "interleaved fused / alone / alone + re-layout, L2 flushed before each",
                      "B": 2, "H": 16, "D": 128, "P": 8, "peak_tflops": peak_tflops,
                      "peak_kind": f"{peak_kind} bf16 burst", "clocks": clocks,
                      "kernel_source": kernel_source_hash()}), flush=True)


def run_tile_spans(args):
    """One launch of the instrumented build (per-tile timestamps) on the workload:
    block period, PV tail, epilogue (the fused stores) and refill per tile."""
    import torch

    import dit_attention_ulysses_gb300 as xs
    from dit_attention_ulysses_gb300 import spans

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = di.WORKLOADS[args.workload]
    q, k, v = (to_device(x, torch, dev) for x in di.random_qkv(w))
    outs = [torch.empty((w.B, w.S // w.P, w.H, w.D), dtype=torch.bfloat16, device=dev) for _ in range(w.P)]
    ws = xs.Workspace.for_shape(w.B, w.S, w.H, w.D, device=dev) if args.schedule == "balanced" else None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    per_cta = -(-w.B * w.H * ((w.S + 127) // 128) // sms) + 2
    for _ in range(3):   # warm-up of the instrumented library, then the recorded launch
        st, ph, ep = spans.record(q, k, v, outs, xs.XS_LAYOUT_A2A, w.scale, per_cta, ws)
    sampler = ClockSampler(0)
    sampler.start()
    t0 = time.time()
    st, ph, ep = spans.record(q, k, v, outs, xs.XS_LAYOUT_A2A, w.scale, per_cta, ws)
    clocks = sampler.stop(t0, time.time())
    ghz = (clocks.get("sm_mhz") or 2070.0) / 1e3
    print(json.dumps({"tile_spans": spans.summarize(st, ghz), "block_phases_cycles": spans.summarize_phases(ph),
                      "epilogue_steps_cycles": spans.summarize_epilogue(ep),
                      "workload": w.name, "sm_ghz_assumed": ghz, "clocks": clocks,
                      "kernel_source": kernel_source_hash()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(di.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", choices=["balanced", "plain"], default="balanced",
                    help="balanced: spread the last partial wave of tiles over all SMs (workspace); "
                         "plain: whole tiles only")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--tile-spans", action="store_true",
                    help="record one launch of the per-tile timestamp build on --workload and print its spans")
    ap.add_argument("--sweep", action="store_true",
                    help="time the sequence sweep (fused, attention alone, attention + re-layout at every S) "
                         "and print it as one JSON record instead of the benchmark line")
    args = ap.parse_args()
    rank, world, local_rank = env_rank()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)   # rank 0 only; other ranks exit without work
        return
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.tile_spans:
        if rank == 0:
            run_tile_spans(args)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")   # barrier and max-over-ranks only; no data-path collective
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
