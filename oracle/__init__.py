"""CPU oracle for fused attention + post-attention Ulysses re-shard.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain fp64 definition that the
CUDA path is checked against; it shares no code with that path.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference legs may import it.  The product package never imports it and has
no CPU fallback.

Source: X-Stage (arXiv 2607.23264), abstract ("tile-granular fusion of the
post-attention All-to-All with FlashAttention" for Ulysses sequence-parallel
attention) and the gist.science technical summary, "Key Contributions" item 3
(FlashAttention-A2A piggybacking).  The pages do not spell out attention
itself; the oracle takes the textbook definition O = softmax(Q K^T * scale) V,
non-causal, no mask, no bias, fp64 throughout (see ``attention_oracle.c``).
``causal=True`` selects the causal variant, which the pages do not treat: row i
attends to keys 0 .. i only (plain attention over the first i + 1 keys).
``attention_varlen`` applies either form to each of several packed sequences.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (brute force, closed forms, invariants, an exact
worked example, an index-coded layout test and a library cross-check).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc + OpenMP (host code, any architecture)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            for suffix in ("", "_causal"):
                f = getattr(lib, "oracle_attention" + suffix)
                f.restype = ctypes.c_int
                f.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, ctypes.c_double, _ptr, ctypes.c_int]
                f = getattr(lib, "oracle_attention_rows" + suffix)
                f.restype = ctypes.c_int
                f.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, ctypes.c_double, _ptr, _ptr, _i64, _ptr,
                              ctypes.c_int]
                f = getattr(lib, "oracle_attention_weights" + suffix)
                f.restype = ctypes.c_int
                f.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, ctypes.c_double, _i64, _i64, _i64, _ptr,
                              _ptr]
            for name in ("oracle_head_shards", "oracle_a2a", "oracle_a2a_inverse"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _i64, _i64]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16)")
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def threads_used(nthreads: int | None = None) -> int:
    """How many OpenMP threads the oracle runs with for ``nthreads``."""
    return _load().oracle_max_threads(nthreads or default_threads())


def _fn(name: str, causal: bool):
    return getattr(_load(), name + ("_causal" if causal else ""))


def attention(q, k, v, scale: float, nthreads: int | None = None, causal: bool = False) -> np.ndarray:
    """Exact attention O [B,S,H,D] (float64) of bf16-bit inputs [B,S,H,D]."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, S, H, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    o = np.empty((B, S, H, D), dtype=np.float64)
    rc = _fn("oracle_attention", causal)(_p(q), _p(k), _p(v), B, S, H, D, float(scale), _p(o),
                                         nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    return o


def attention_rows(q, k, v, scale: float, rows_b, rows_s, nthreads: int | None = None,
                   causal: bool = False) -> np.ndarray:
    """Exact attention of selected query rows: returns [n_rows, H, D] float64."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, S, H, D = q.shape
    rb = np.ascontiguousarray(rows_b, dtype=np.int64)
    rs = np.ascontiguousarray(rows_s, dtype=np.int64)
    o = np.empty((len(rb), H, D), dtype=np.float64)
    rc = _fn("oracle_attention_rows", causal)(_p(q), _p(k), _p(v), B, S, H, D, float(scale),
                                              _p(rb), _p(rs), len(rb), _p(o),
                                              nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    return o


def attention_weights(q, k, v, scale: float, b: int, i: int, h: int, causal: bool = False):
    """Normalised softmax weights w[S] and output row o[D] of query (b, i, h)
    (causal: w[j] = 0 for j > i)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, S, H, D = q.shape
    w = np.empty(S, dtype=np.float64)
    o = np.empty(D, dtype=np.float64)
    rc = _fn("oracle_attention_weights", causal)(_p(q), _p(k), _p(v), B, S, H, D, float(scale),
                                                 b, i, h, _p(w), _p(o))
    if rc != 0:
        raise RuntimeError("oracle_attention_weights failed")
    return w, o


def head_shards(o: np.ndarray, P: int) -> np.ndarray:
    """O [B,S,H,D] -> the P Ulysses head shards, [P, B, S, H/P, D]."""
    o = np.ascontiguousarray(o, dtype=np.float64)
    B, S, H, D = o.shape
    L = np.empty((P, B, S, H // P, D), dtype=np.float64)
    if _load().oracle_head_shards(_p(o), _p(L), B, S, H, D, P) != 0:
        raise ValueError("head_shards needs H % P == 0")
    return L


def a2a(L: np.ndarray) -> np.ndarray:
    """Post-attention All-to-All: head shards [P,B,S,H/P,D] -> sequence shards [P,B,S/P,H,D]."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    P, B, S, Hl, D = L.shape
    out = np.empty((P, B, S // P, Hl * P, D), dtype=np.float64)
    if _load().oracle_a2a(_p(L), _p(out), B, S, Hl * P, D, P) != 0:
        raise ValueError("a2a needs S % P == 0")
    return out


def a2a_inverse(out: np.ndarray) -> np.ndarray:
    """Inverse exchange: sequence shards [P,B,S/P,H,D] -> head shards [P,B,S,H/P,D]."""
    out = np.ascontiguousarray(out, dtype=np.float64)
    P, B, Sl, H, D = out.shape
    L = np.empty((P, B, Sl * P, H // P, D), dtype=np.float64)
    if _load().oracle_a2a_inverse(_p(out), _p(L), B, Sl * P, H, D, P) != 0:
        raise ValueError("a2a_inverse needs H % P == 0")
    return L


def attention_a2a(q, k, v, scale: float, P: int, nthreads: int | None = None, causal: bool = False) -> np.ndarray:
    """The whole oracle path: attention, then the explicit Ulysses re-shard.

    Returns the P output shards as one array [P, B, S/P, H, D] (float64).
    """
    return a2a(head_shards(attention(q, k, v, scale, nthreads, causal), P))


def attention_varlen(q, k, v, seqlens, scale: float, causal: bool = False,
                     nthreads: int | None = None) -> np.ndarray:
    """Attention of packed variable-length sequences (not on the pages; the packed
    batches of variable-length attention kernels): q, k, v are [1, T, H, D] bf16
    bits holding sequences of lengths ``seqlens`` back to back (T = sum of them),
    and every query row attends only to the keys of its own sequence (causal: of
    its own sequence and at or before its own position).  Computed as exact
    attention of each sequence's slice on its own.  Returns [1, T, H, D] float64."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    lens = [int(n) for n in seqlens]
    if q.ndim != 4 or q.shape[0] != 1 or any(n < 0 for n in lens) or sum(lens) != q.shape[1]:
        raise ValueError("packed inputs are [1, T, H, D] with T = sum(seqlens), seqlens >= 0")
    o = np.empty(q.shape, dtype=np.float64)
    start = 0
    for n in lens:
        if n:
            sl = slice(start, start + n)
            o[:, sl] = attention(q[:, sl], k[:, sl], v[:, sl], scale, nthreads, causal)
        start += n
    return o


def _exact_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 values that are exactly bf16 -> their bf16 bit patterns (checked)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    back = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if not np.array_equal(back, f):
        raise ValueError("values are not exactly representable in bf16")
    return bits


def ulysses_attention(q_shards, k_shards, v_shards, scale: float, nthreads: int | None = None) -> np.ndarray:
    """The Ulysses attention step of P ranks, in its three steps (DeepSpeed-Ulysses
    sequence parallelism, as used by the X-Stage paper's DiT inference):

    1. pre-attention All-to-All: rank p's sequence shard [B,S/P,H,D] of each of Q, K, V
       is exchanged so that rank r holds all S rows of heads [r*H/P, (r+1)*H/P);
    2. every rank runs exact attention on its own heads;
    3. post-attention All-to-All back to sequence shards.

    q_shards etc.: [P, B, S/P, H, D] bf16 bits (uint16).  Returns [P, B, S/P, H, D] float64.
    """
    widen = lambda b: (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)
    Lq, Lk, Lv = (a2a_inverse(widen(x)) for x in (q_shards, k_shards, v_shards))
    O = np.stack([attention(_exact_bf16_bits(Lq[r]), _exact_bf16_bits(Lk[r]), _exact_bf16_bits(Lv[r]), scale,
                            nthreads) for r in range(Lq.shape[0])])
    return a2a(O)
