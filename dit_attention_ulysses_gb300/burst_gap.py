"""Burst-Gap model of the store path: measurement driver and fit.

X-Stage (arXiv 2607.23264), gist.science technical summary, "Methodology: The
X-Stage Abstraction and Burst-Gap Model": K producers issue bursts of stores of
aggregate volume V separated by a producer-side gap G, and the sender-visible
issue time of a burst is

    T_iss(G; K, V) = max(T0_iss(K, V), V / R - G)

with T0_iss the backpressure-free issue time, R the effective drain rate and Q
the effective outstanding capacity ("the finite volume that can remain
outstanding before the issue rate stalls").

The pages give no formula for Q or for the shape of T0_iss.  Readings used here:

* for a fixed number of producers T0_iss is affine in the volume,
  T0(V) = t_fix + V / B0 (a fixed per-burst cost and an issue bandwidth B0);
* a queue model of the path: the producers issue at B0 while the outstanding
  volume x is below Q and at the drain rate R once it has reached Q; the path
  drains at R whenever x > 0, during bursts and gaps alike.  Its periodic
  steady state is exactly the pages' formula as long as one burst's net
  accumulation V (1 - R/B0) fits in Q (Q then only sets how many bursts it
  takes to get there; a larger burst is drain-limited beyond Q even when
  isolated), so
    - R follows from back-to-back bursts (G = 0): R = V / T_iss;
    - Q follows from the transient: started from an empty path, bursts run at
      T0 until the accumulated outstanding volume, V - R T0 per burst net of
      drain, reaches Q.

On one GPU the path is the fused epilogue's: SM -> L2 -> HBM, into a buffer
larger than L2 (the pages measure remote NVLink stores: R ~ 717 GB/s there).
The kernel is ``xs_burst_gap`` (csrc/burst_gap.cu); this module drives it and
fits its issue times.  ``python -m dit_attention_ulysses_gb300.burst_gap`` runs
the default sweeps and prints one JSON line.
"""
from __future__ import annotations

import json
from dataclasses import dataclass

import numpy as np

__all__ = ["BurstGapParams", "t0", "steady_state", "simulate", "fit_t0", "drain_rate", "capacity_from_transient",
           "measure", "main"]


@dataclass
class BurstGapParams:
    t_fix_ns: float   # fixed per-burst issue cost
    b0_gbs: float     # backpressure-free issue bandwidth (bytes per ns = GB/s), all producers
    r_gbs: float      # drain rate
    q_bytes: float    # outstanding capacity


def t0(p: BurstGapParams, V):
    """Backpressure-free issue time (ns) of a burst of V bytes."""
    return p.t_fix_ns + np.asarray(V, dtype=np.float64) / p.b0_gbs


def steady_state(p: BurstGapParams, V, G):
    """The pages' formula: issue time (ns) of periodic bursts of V bytes with gap G (ns)."""
    return np.maximum(t0(p, V), np.asarray(V, dtype=np.float64) / p.r_gbs - np.asarray(G, dtype=np.float64))


def simulate(p: BurstGapParams, V: float, G: float, bursts: int, x0: float = 0.0):
    """Issue times (ns) of ``bursts`` consecutive bursts of V bytes with gap G
    under the queue model, starting with x0 bytes outstanding (0: an idle path).
    The fixed cost t_fix is charged as issue time without stores."""
    x = float(x0)
    out = []
    for _ in range(bursts):
        t = p.t_fix_ns
        x = max(0.0, x - p.r_gbs * p.t_fix_ns)
        left = float(V)
        if x < p.q_bytes:
            # phase 1: issue at B0 while x grows at B0 - R, up to Q or to the end of the burst
            grow = p.b0_gbs - p.r_gbs
            t1 = left / p.b0_gbs if grow <= 0 else min(left / p.b0_gbs, (p.q_bytes - x) / grow)
            t += t1
            left -= p.b0_gbs * t1
            x = max(0.0, x + grow * t1)
        if left > 1e-6:
            t += left / p.r_gbs   # phase 2: issue throttled to the drain, x stays at Q
        out.append(t)
        x = max(0.0, x - p.r_gbs * G)   # the gap drains
    return np.array(out)


def fit_t0(V, T):
    """Least squares T = t_fix + V / B0 with relative weights; returns (t_fix, B0, rms_rel_err)."""
    V = np.asarray(V, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    w = 1.0 / T
    A = np.stack([np.ones_like(V), V], axis=1) * w[:, None]
    (a, b), *_ = np.linalg.lstsq(A, T * w, rcond=None)
    pred = a + b * V
    return float(a), float(1.0 / b), float(np.sqrt(np.mean(((pred - T) / T) ** 2)))


def drain_rate(V: float, T_back_to_back: float) -> float:
    """R (GB/s) from the steady-state issue time of back-to-back bursts (G = 0)."""
    return float(V) / float(T_back_to_back)


def capacity_from_transient(V: float, T, t0_ns: float, r_gbs: float, tol: float = 0.1):
    """Bounds (bytes) on Q from the issue times of back-to-back bursts started on
    an idle path.  Each stall-free burst leaves V - R T0 bytes more outstanding;
    let n be the index of the first burst slower than (1 + tol) T0.  Burst n
    reached Q, and burst n - 1 may have touched it without showing (a stall
    shorter than tol T0), so (n - 1)(V - R T0) <= Q < (n + 1)(V - R T0).
    Upper bound infinite if no burst stalled."""
    T = np.asarray(T, dtype=np.float64)
    per = float(V) - r_gbs * t0_ns
    if per <= 0:
        return (float("inf"), float("inf"))
    slow = np.nonzero(T > (1.0 + tol) * t0_ns)[0]
    if slow.size == 0:
        return (max(0, T.size - 1) * per, float("inf"))
    n = int(slow[0])
    return (max(0, n - 1) * per, (n + 1) * per)


def measure(dst, producers: int, volumes, gap_ns: int, bursts: int = 24, skip: int = 4, stream=None, raw=False,
            lead_ns: int = 0):
    """Sender-visible issue time (ns) of bursts: per burst the maximum over the
    producers (a burst is issued when its slowest producer is done); per volume
    the median over the bursts after the first ``skip`` (raw=True: the issue
    times of all bursts of the first volume)."""
    import torch
    import dit_attention_ulysses_gb300 as xs
    out = []
    for V in volumes:
        t = xs.xs_burst_gap(dst, producers, int(V), bursts, int(gap_ns), stream, lead_ns=int(lead_ns))
        torch.cuda.synchronize()
        per_burst = t.max(dim=1).values.cpu().numpy().astype(np.float64)
        if raw:
            return per_burst
        out.append(float(np.median(per_burst[skip:])))
    return out


def main(argv=None) -> int:
    import argparse
    import torch
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--producers", type=int, default=0, help="K (default: the SM count)")
    ap.add_argument("--dst-mib", type=int, default=4096, help="destination buffer (MiB), larger than L2")
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    K = args.producers or torch.cuda.get_device_properties(dev).multi_processor_count
    dst = torch.empty(args.dst_mib << 20, dtype=torch.uint8, device=dev)
    # 1. isolated bursts (a 2 ms gap before each): T0 over per-producer volumes
    #    4 KiB .. 16 MiB, fitted above the timer/barrier floor
    max_per = (args.dst_mib << 20) // K
    per = [p for p in (4096 * 2 ** i for i in range(13)) if p <= max_per]
    vols = [p * K for p in per]
    t_iso = measure(dst, K, vols, gap_ns=2_000_000, bursts=8, skip=2)
    floor = min(t_iso)
    keep = [i for i, t in enumerate(t_iso) if t >= 4 * floor]
    t_fix, b0, t0_err = fit_t0([vols[i] for i in keep], [t_iso[i] for i in keep])
    # 2. back-to-back bursts of 1 MiB per producer: the drain rate
    V = 1048576 * K
    t_b2b = measure(dst, K, [V], gap_ns=0, bursts=32, skip=8)[0]
    r = drain_rate(V, t_b2b)
    p = BurstGapParams(t_fix_ns=t_fix, b0_gbs=b0, r_gbs=r, q_bytes=float("nan"))
    t0_v = float(t0(p, V))
    # 3. the transient from a drained path (a 2 ms in-kernel lead-in spin, which
    #    keeps the clocks up, unlike an idle GPU): the capacity
    t_tr = measure(dst, K, [V], gap_ns=0, bursts=16, raw=True, lead_ns=2_000_000)
    q_lo, q_hi = capacity_from_transient(V, t_tr, t0_v, r)
    # 4. gap sweep at the same volume against the pages' steady-state formula
    gaps = [int(max(0.0, V / r - t0_v) * f) for f in (0.0, 0.15, 0.3, 0.5, 0.7, 1.0, 1.5)]
    t_gap = [measure(dst, K, [V], gap_ns=G, bursts=32, skip=8)[0] for G in gaps]
    model = steady_state(p, V, gaps)
    line = {"metric": "burst_gap_fit", "producers": K, "dst_bytes": args.dst_mib << 20,
            "t_fix_ns": t_fix, "b0_gbs": b0, "t0_fit_rms_rel_err": t0_err, "r_gbs": r,
            "q_bytes_bounds": [q_lo, q_hi], "timer_floor_ns": floor,
            "isolated": {"volume_bytes": vols, "issue_ns": t_iso, "fitted": keep},
            "transient": {"volume_bytes": V, "issue_ns": [float(x) for x in t_tr]},
            "steady_state": {"volume_bytes": V, "t0_ns": t0_v, "gap_ns": gaps, "issue_ns": t_gap,
                             "model_ns": [float(x) for x in model],
                             "rms_rel_err": float(np.sqrt(np.mean(((model - np.array(t_gap)) / np.array(t_gap)) ** 2)))}}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
