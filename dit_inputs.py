"""Seeded synthetic inputs for the fused attention + Ulysses re-shard path.

This module is the only code shared by the CUDA path's tests/bench and by the
CPU oracle.  It holds no attention arithmetic: it draws bf16 tensors of the DiT
workload shapes, builds the index-coded inputs of the layout test, and names the
workloads.  Everything it returns is raw bf16 bit patterns (``numpy.uint16``) in
the ``[B, S, H, D]`` layout (D fastest), so each side converts them itself.

Sampling recipe (fixed here so that both sides see identical data):

* N(0,1) entries: ``numpy.random.Generator(PCG64)`` float32 standard normals,
  rounded to bf16 with round-to-nearest-even.  The three streams for Q, K and V
  come from ``SeedSequence(seed).spawn(4)[0..2]``.
* Outlier channels (the large video-DiT workload): per head, 4 of the D channels
  are drawn without replacement from stream ``spawn(4)[3]``; the same channels are
  used for Q, K and V and for every batch entry; the float32 sample is multiplied
  by 8 before the bf16 rounding.
* The index-coded layout input (``layout_code_inputs``) is exact: every value is
  +-1 or a small integer, all representable in bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "SWEEP_S",
    "sweep_workload",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "random_qkv",
    "outlier_channels",
    "layout_code_inputs",
    "layout_code_value",
    "sample_rows",
]


@dataclass(frozen=True)
class Workload:
    """One DiT attention workload: shapes, virtual-rank count and input recipe."""

    name: str
    B: int
    H: int
    S: int
    D: int
    P: int
    scale: float
    outliers: int = 0          # channels per head scaled by ``outlier_gain``
    outlier_gain: float = 8.0
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        """Tensor FLOPs of non-causal attention: 2*S*S*D for QK^T plus the same for PV."""
        return 4 * self.B * self.H * self.S * self.S * self.D

    @property
    def tensor_bytes(self) -> int:
        return self.B * self.S * self.H * self.D * 2


# Sequence lengths of the B=2, H=16, P=8 sweep: doubling from 1024 to 131072.
SWEEP_S = [1024 * (1 << i) for i in range(8)]


def sweep_workload(S: int) -> Workload:
    return Workload(f"sweep_S{S}", B=2, H=16, S=S, D=128, P=8,
                    scale=1.0 / math.sqrt(128), note="sequence sweep point")


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, S=256, D=64, P=2, scale=1.0 / math.sqrt(64),
                     note="correctness case, 2 shards of [1,128,2,64]"),
    "image": Workload("image", B=1, H=24, S=4608, D=128, P=4, scale=1.0 / math.sqrt(128),
                      note="image-DiT shape, 4 shards of [1,1152,24,128]"),
    "video_small": Workload("video_small", B=1, H=12, S=32768, D=128, P=4,
                            scale=1.0 / math.sqrt(128),
                            note="video-DiT small, 4 shards of [1,8192,12,128]"),
    "video_large": Workload("video_large", B=1, H=40, S=75776, D=128, P=8,
                            scale=1.0 / math.sqrt(128), outliers=4,
                            note="video-DiT large with outlier channels, 8 shards of [1,9472,40,128]"),
    # head dimension 64 at the small video model's width (24 x 64 = 12 x 128)
    "video_small_d64": Workload("video_small_d64", B=1, H=24, S=32768, D=64, P=4,
                                scale=1.0 / math.sqrt(64),
                                note="video-DiT small, 24 heads of 64, 4 shards of [1,8192,24,64]"),
}
for _s in SWEEP_S:
    WORKLOADS[f"sweep_S{_s}"] = sweep_workload(_s)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits.

    Finite inputs only (the generators never produce NaN/Inf).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(w: Workload) -> np.ndarray:
    """Per-head outlier channel indices, shape [H, outliers], sorted within a head."""
    if w.outliers == 0:
        return np.zeros((w.H, 0), dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(w.seed).spawn(4)[3]))
    return np.stack([np.sort(rng.choice(w.D, size=w.outliers, replace=False)) for _ in range(w.H)])


def random_qkv(w: Workload, S: int | None = None):
    """Seeded bf16 Q, K, V of shape [B, S, H, D] as uint16 bit arrays.

    ``S`` overrides the workload's sequence length (used for small parity cases
    with the same recipe).
    """
    S = w.S if S is None else S
    shape = (w.B, S, w.H, w.D)
    seqs = np.random.SeedSequence(w.seed).spawn(4)
    chans = outlier_channels(w)
    out = []
    for i in range(3):
        rng = np.random.Generator(np.random.PCG64(seqs[i]))
        x = rng.standard_normal(shape, dtype=np.float32)
        if w.outliers:
            for h in range(w.H):
                x[:, :, h, chans[h]] *= np.float32(w.outlier_gain)
        out.append(f32_to_bf16_bits(x))
        del x
    return tuple(out)


# ----------------------------------------------------------------------------
# Index-coded inputs for the bit-exact layout test.
#
# Q = K carry a +-1 code of the sequence index: bit i of s (i < nbits) is
# repeated over REP consecutive channels as (+1 if the bit is 1 else -1); the
# remaining channels are +1.  Then q_s . k_t = D - 2*REP*hamming(s, t), so the
# own key beats every other key by at least 2*REP.  With a large scale the
# softmax row is one-hot at t = s, and O[b,s,h,:] = V[b,s,h,:].
# V carries the index of its own row: channel 0 = s mod 256, 1 = s // 256 mod 256,
# 2 = h, 3 = b, channels d >= 4 hold d mod 256.  All are integers < 256 and
# exact in bf16.
# ----------------------------------------------------------------------------
LAYOUT_REP = 7
LAYOUT_REP_MIN = 4   # where 7 repeats per bit do not fit D (long sequences at D = 64)


def _layout_nbits(S: int) -> int:
    return max(1, math.ceil(math.log2(S))) if S > 1 else 1


def _layout_rep(S: int, D: int) -> int:
    """Channels per code bit: 7 where they fit, else 4 (the own key then beats
    every other by at least 8 in q.k, and the second-best weight is exp(-16*8)
    relative to it, still far below fp32 resolution)."""
    nbits = _layout_nbits(S)
    for r in (LAYOUT_REP, LAYOUT_REP_MIN):
        if nbits * r <= D:
            return r
    raise ValueError(f"S={S} needs {nbits * LAYOUT_REP_MIN} code channels > D={D}")


def layout_code_value(b: int, s: np.ndarray | int, h: int, D: int) -> np.ndarray:
    """Expected bf16-exact V row (as float32) for index (b, s, h): shape [..., D]."""
    s = np.asarray(s)
    row = np.empty(s.shape + (D,), dtype=np.float32)
    row[...] = (np.arange(D) % 256).astype(np.float32)
    row[..., 0] = (s % 256).astype(np.float32)
    row[..., 1] = ((s // 256) % 256).astype(np.float32)
    row[..., 2] = float(h % 256)
    row[..., 3] = float(b % 256)
    return row


def layout_code_inputs(B: int, S: int, H: int, D: int):
    """(q, k, v, scale) bf16 bit arrays for the one-hot layout test.

    Each bit of s takes 7 channels where ceil(log2 S) * 7 <= D (S <= 2**18 at
    D = 128, S <= 2**9 at D = 64), else 4 (S <= 2**16 at D = 64).  The returned
    scale (16) makes the second-best key's weight exp(-16*14), or exp(-16*8)
    with 4 channels per bit, relative to the own key: far below fp32 resolution.
    """
    nbits = _layout_nbits(S)
    r = _layout_rep(S, D)
    s = np.arange(S)
    code = np.ones((S, D), dtype=np.float32)
    for i in range(nbits):
        bit = ((s >> i) & 1).astype(np.float32) * 2.0 - 1.0
        code[:, i * r:(i + 1) * r] = bit[:, None]
    qk = np.broadcast_to(code[None, :, None, :], (B, S, H, D))
    q = f32_to_bf16_bits(qk)
    k = q.copy()
    v = np.empty((B, S, H, D), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            v[b, :, h, :] = layout_code_value(b, s, h, D)
    return q, k, f32_to_bf16_bits(v), 16.0


def sample_rows(w: Workload, n: int, seed: int = 1, S: int | None = None):
    """Seeded sample of about n distinct (b, s) query rows, sorted.

    Always includes the first and last row of every shard of every batch entry
    (the shard boundaries); the rest are drawn uniformly without replacement.
    Returns two int64 arrays (b, s).
    """
    S = w.S if S is None else S
    total = w.B * S
    shard = S // w.P
    forced = set()
    for b in range(w.B):
        for p in range(w.P):
            forced.add(b * S + p * shard)
            forced.add(b * S + p * shard + shard - 1)
    forced = {x for x in forced if 0 <= x < total}
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed + 1000)))
    want = max(0, min(n, total) - len(forced))
    picked = set(forced)
    while len(picked) < len(forced) + want:
        for x in rng.integers(0, total, size=2 * want + 8):
            if len(picked) >= len(forced) + want:
                break
            picked.add(int(x))
    arr = np.array(sorted(picked), dtype=np.int64)
    return arr // S, arr % S


def layout_code_inputs_torch(B: int, S: int, H: int, D: int, device="cuda"):
    """The same index-coded (q, k, v, scale) as ``layout_code_inputs``, built
    directly as bf16 torch tensors on ``device`` (for full-size cases, where the
    NumPy construction would be slow).  Exact: every value is +-1 or an integer
    below 256."""
    import torch
    nbits = _layout_nbits(S)
    r = _layout_rep(S, D)
    s = torch.arange(S, device=device, dtype=torch.int64)
    code = torch.ones((S, D), device=device, dtype=torch.float32)
    for i in range(nbits):
        bit = ((s >> i) & 1).to(torch.float32) * 2.0 - 1.0
        code[:, i * r:(i + 1) * r] = bit[:, None]
    q = code.to(torch.bfloat16)[None, :, None, :].expand(B, S, H, D).contiguous()
    k = q.clone()
    v = layout_code_value_torch(B, S, H, D, device)
    return q, k, v, 16.0


def layout_code_value_torch(B: int, S: int, H: int, D: int, device="cuda", s_offset: int = 0, S_rows=None):
    """bf16 tensor [B, S_rows, H, D] holding the index code of rows
    s_offset .. s_offset + S_rows - 1 (see ``layout_code_value``)."""
    import torch
    n = S if S_rows is None else S_rows
    s = torch.arange(s_offset, s_offset + n, device=device, dtype=torch.int64)
    v = (torch.arange(D, device=device, dtype=torch.int64) % 256).to(torch.float32)
    v = v.expand(B, n, H, D).clone()
    v[..., 0] = (s % 256).to(torch.float32)[None, :, None]
    v[..., 1] = ((s // 256) % 256).to(torch.float32)[None, :, None]
    v[..., 2] = (torch.arange(H, device=device) % 256).to(torch.float32)[None, None, :]
    v[..., 3] = (torch.arange(B, device=device) % 256).to(torch.float32)[:, None, None]
    return v.to(torch.bfloat16)
