"""Per-tile timestamps of the attention kernel: where a tile's time goes.

X-Stage (gist.science technical summary, "Results") reads the fused kernel's
behaviour from per-tile store spans.  This module runs the attention kernel from
a separately built library, ``libxsattn_spans.so`` (the same sources compiled
with ``XS_TILE_SPANS``; the product library has no stamps), in which warp 0 of
every CTA records six words per piece of work:

  0  %globaltimer (ns) when the piece's first scores are seen
  1  clock64 at the same moment
  2  clock64 when the piece's last P is written to tensor memory
  3  clock64 when its last PV has completed (the epilogue may start)
  4  clock64 after the epilogue's stores to the owner's shard are issued
  5  (key blocks << 32) | piece kind (0 whole tile, 1 head of a split tile, 2 part)

``summarize`` turns a recording into per-tile spans in SM cycles and
microseconds: the block period (first scores to last P, per key block), the PV
tail (last P to last PV done), the epilogue span (last PV done to stores
issued: the fused All-to-All's cost on the critical path) and the refill (stores
issued to the next piece's first scores in the same CTA).

For the first piece of every CTA and its key blocks PHASE_J0 .. PHASE_J0 +
PHASE_BLOCKS - 1 (past the launch's pipeline fill) the build also records
PHASE_WORDS clock64 stamps per block: the softmax's steps (warp 0,
lane 0: 0 before the scores wait, 1 scores seen, 2 scores loaded from tensor
memory, 3 row max combined, 4 exponentials done, 5 O rescaled if it had to be, 6 P stored and
signalled), the S issuer (11 buffer free seen, 12 K tile seen, 7 S MMAs issued), the
PV issuer (9 P seen, 10 V tile seen, 8 PV MMAs issued), the producer (13 K tile
load issued, 14 V tile load issued) and lane 0 of every softmax warp w (16 + w: P
stored and signalled; warp w runs on sub-partition w % 4, beside warp w + 4 and
one of the single-thread roles or the idle warp).
``summarize_phases`` gives the median duration of each step.

Last, EPI_WORDS stamps per CTA of warp 0's epilogue of its first piece (when it
is a whole tile): 0 last PV seen done, 1 destination row computed, then for each
32-column chunk of the thread's half row (two at D = 128) its O loaded from
tensor memory, its bf16 values staged in shared memory and its global stores
issued.  ``summarize_epilogue`` gives the median of each step.
"""
from __future__ import annotations

import ctypes

import numpy as np

SPAN_WORDS = 6
PHASE_J0 = 8
PHASE_BLOCKS = 32
PHASE_WORDS = 24
EPI_WORDS = 8


def parse(stamps: np.ndarray) -> list[dict]:
    """Recorded words [grid, per_cta, 6] (uint64) -> one dict per recorded piece, in
    CTA order and piece order, with the raw stamps, the CTA and the piece index."""
    stamps = np.asarray(stamps, dtype=np.uint64)
    out = []
    for cta in range(stamps.shape[0]):
        for k in range(stamps.shape[1]):
            w = [int(x) for x in stamps[cta, k]]
            if w[5] == 0:
                continue
            out.append({"cta": cta, "piece": k, "blocks": w[5] >> 32, "kind": w[5] & 0xFFFFFFFF,
                        "t_ns": w[0], "c_first": w[1], "c_last_p": w[2], "c_o_done": w[3], "c_stored": w[4]})
    return out


def _stats(x):
    x = np.asarray(x, dtype=np.float64)
    if x.size == 0:
        return None
    p10, p50, p90 = np.percentile(x, [10, 50, 90])
    return {"p10": float(p10), "p50": float(p50), "p90": float(p90), "n": int(x.size)}


def summarize(stamps: np.ndarray, sm_ghz: float) -> dict:
    """Spans of every recorded piece (cycles, and microseconds at sm_ghz):
    block period, PV tail, epilogue (store) span and refill, as p10/p50/p90."""
    recs = parse(stamps)
    per_block, tail, epi, refill = [], [], [], []
    by_cta = {}
    for r in recs:
        by_cta.setdefault(r["cta"], []).append(r)
        if r["blocks"] > 1:
            per_block.append((r["c_last_p"] - r["c_first"]) / (r["blocks"] - 1))
        tail.append(r["c_o_done"] - r["c_last_p"])
        epi.append(r["c_stored"] - r["c_o_done"])
    for rs in by_cta.values():
        rs.sort(key=lambda r: r["piece"])
        for a, b in zip(rs, rs[1:]):
            if b["piece"] == a["piece"] + 1:
                refill.append(b["c_first"] - a["c_stored"])
    to_us = lambda s: None if s is None else {k: (v / (sm_ghz * 1e3) if k != "n" else v) for k, v in s.items()}
    cyc = {"block_period": _stats(per_block), "pv_tail": _stats(tail), "epilogue": _stats(epi),
           "refill": _stats(refill)}
    starts = [r["t_ns"] for r in recs]
    return {"pieces": len(recs), "ctas": len(by_cta), "cycles": cyc, "us": {k: to_us(v) for k, v in cyc.items()},
            "first_to_last_start_us": (max(starts) - min(starts)) / 1e3 if starts else None}


def summarize_phases(phases: np.ndarray, first_block: int = 0) -> dict:
    """Block-phase stamps [grid, PHASE_BLOCKS, PHASE_WORDS] -> median cycles of each
    softmax step over the recorded blocks >= first_block of every CTA."""
    ph = np.asarray(phases, dtype=np.int64)
    rows = []
    for cta in range(ph.shape[0]):
        for j in range(first_block, ph.shape[1] - 1):
            a, b = ph[cta, j], ph[cta, j + 1]
            if a[0] == 0 or a[6] == 0 or b[0] == 0:
                continue
            rows.append({"wait_scores": a[1] - a[0], "load_scores": a[2] - a[1], "row_max": a[3] - a[2],
                         "exponentials": a[4] - a[3], "rescale_o": a[5] - a[4], "store_p": a[6] - a[5],
                         "to_next_block": b[0] - a[6], "period": b[0] - a[0],
                         "s_issued_to_seen": a[1] - a[7], "p_signalled_to_pv_issued": a[8] - a[6],
                         **{f"warp{w}_p_signalled_after_warp0": a[16 + w] - a[16] for w in range(1, 8)},
                         "pv_sees_p_after_warp0": a[9] - a[6], "pv_sees_v_after_p": a[10] - a[9],
                         "pv_issue_after_v": a[8] - a[10], "v_load_to_seen": a[10] - a[14],
                         "s_buffer_free_after_softmax_start": a[11] - a[0], "s_sees_k_after_free": a[12] - a[11],
                         "s_issue_after_k": a[7] - a[12], "k_load_to_seen": a[12] - a[13]})
    if not rows:
        return {"blocks": 0}
    out = {"blocks": len(rows)}
    for k in rows[0]:
        out[k] = float(np.median([r[k] for r in rows]))
    return out


def summarize_epilogue(epi: np.ndarray) -> dict:
    """Epilogue stamps [grid, EPI_WORDS] -> median cycles of each step over the CTAs
    whose first piece ended in a whole-tile epilogue."""
    e = np.asarray(epi, dtype=np.int64)
    names = ["destination_row", "load_o_0", "stage_0", "stores_0", "load_o_1", "stage_1", "stores_1"]
    rows = [r for r in e if r[0] != 0 and r[4] != 0]
    if not rows:
        return {"ctas": 0}
    out = {"ctas": len(rows)}
    for i, k in enumerate(names):
        d = [r[i + 1] - r[i] for r in rows if r[i + 1] != 0]
        if d:
            out[k] = float(np.median(d))
    last = [r[max(i for i in range(EPI_WORDS) if r[i] != 0)] - r[0] for r in rows]
    out["total"] = float(np.median(last))
    return out


def load():
    """The instrumented library (built here if needed), with the entry points used."""
    from . import _build
    path = _build.build(variant="spans")
    lib = ctypes.CDLL(path)
    lib.xs_attn_set_tile_spans.restype = ctypes.c_int
    lib.xs_attn_set_tile_spans.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    lib.xs_attn_fwd_balanced.restype = ctypes.c_int
    lib.xs_attn_fwd_balanced.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)] + \
        [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.xs_attn_get_device_error.restype = ctypes.c_int
    lib.xs_attn_get_device_error.argtypes = [ctypes.c_void_p]
    return lib


def record(q, k, v, outs, layout: int, scale: float, per_cta: int, workspace=None):
    """One launch of the instrumented kernel (xs_attn_fwd_balanced's arguments, torch
    tensors on the current device); returns the stamps [grid, per_cta, 6], the
    block-phase stamps [grid, PHASE_BLOCKS, PHASE_WORDS] and the epilogue stamps
    [grid, EPI_WORDS], all uint64."""
    import torch
    lib = load()
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    n_spans = sms * per_cta * SPAN_WORDS
    n_phase = sms * PHASE_BLOCKS * PHASE_WORDS
    buf = torch.zeros(n_spans + n_phase + sms * EPI_WORDS, dtype=torch.int64, device=q.device)
    if lib.xs_attn_set_tile_spans(buf.data_ptr(), sms, per_cta) != 0:
        raise RuntimeError("xs_attn_set_tile_spans failed")
    B, S, H, D = q.shape
    ptrs = (ctypes.c_void_p * len(outs))(*[o.data_ptr() for o in outs])
    wp, wn = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.xs_attn_fwd_balanced(q.data_ptr(), k.data_ptr(), v.data_ptr(), layout, ptrs, B, S, H, D, len(outs),
                                  scale, wp, wn, stream)
    if rc != 0 or lib.xs_attn_get_device_error(stream) != 0:
        raise RuntimeError(f"instrumented launch failed ({rc})")
    lib.xs_attn_set_tile_spans(None, 0, 0)
    words = buf.cpu().numpy().view(np.uint64)
    return (words[:n_spans].reshape(sms, per_cta, SPAN_WORDS),
            words[n_spans:n_spans + n_phase].reshape(sms, PHASE_BLOCKS, PHASE_WORDS),
            words[n_spans + n_phase:].reshape(sms, EPI_WORDS))
