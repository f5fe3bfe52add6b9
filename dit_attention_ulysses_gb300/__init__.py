"""Fused sequence-parallel attention + Ulysses All-to-All layout for GB300.

Python binding of ``libxsattn.so`` (hand-written sm_103a CUDA kernels behind a
C ABI, declared in ``include/xsattn.h``).  This module only marshals
arguments: it turns torch tensors into pointers and sizes, picks the current
CUDA stream, and raises :class:`XsError` on a non-zero return code.  Every
step of the computation runs in the library's kernels; there is no fallback.
PyTorch is used for device memory and streams only.

Method: X-Stage (arXiv 2607.23264), abstract and the gist.science technical
summary, "Key Contributions" item 3: the attention output-tile owner stores
each finished tile straight into the post-attention Ulysses All-to-All layout
(the sequence shard of the rank that owns the tile's rows) and resumes its next
tile.  On one GPU the P ranks are P device buffers.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "XsError",
    "lib",
    "xs_attn_a2a_fwd",
    "xs_attn_fwd",
    "xs_attn_heads_fwd",
    "xs_relayout_a2a",
    "xs_relayout_a2a_inverse",
    "xs_attn_ulysses_fwd",
    "xs_attn_ulysses_rank_fwd",
    "xs_burst_gap",
    "xs_attn_a2a_fwd_staged",
    "xs_attn_workspace_bytes",
    "xs_attn_fwd_balanced",
    "xs_attn_fwd_balanced_noalloc",
    "xs_attn_causal_fwd",
    "xs_attn_varlen_fwd",
    "Workspace",
    "xs_attn_get_device_error",
    "xs_attn_get_device_error_info",
    "xs_attn_error_string",
    "attn_a2a",
    "LIB_PATH",
    "EXPORTS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libxsattn.so")

# Error codes of include/xsattn.h
XS_OK = 0
XS_ERR_NULL = -1
XS_ERR_SHAPE = -2
XS_ERR_HEAD_DIM = -3
XS_ERR_DIVISIBILITY = -4
XS_ERR_TOO_MANY_RANKS = -5
XS_ERR_ALIGNMENT = -6
XS_ERR_OVERLAP = -7
XS_ERR_SCALE = -8
XS_ERR_CUDA = -9
XS_ERR_DEVICE_TIMEOUT = -10
XS_ERR_UNSUPPORTED_DEVICE = -11
XS_ERR_WORKSPACE = -12
XS_ERR_LAYOUT = -13
XS_ERR_DEVICE_DRAIN = -14
XS_ERR_DEVICE_BOUNDS = -15
XS_ERR_UNAVAILABLE = -16
XS_MAX_P = 16
XS_LAYOUT_A2A = 0
XS_LAYOUT_CONTIGUOUS = 1
XS_LAYOUT_HEADS = 2

_vp = ctypes.c_void_p
_int = ctypes.c_int
_f32 = ctypes.c_float
_size = ctypes.c_size_t

# name -> (restype, argtypes); the full exported C ABI
EXPORTS = {
    "xs_attn_a2a_fwd": (_int, [_vp, _vp, _vp, ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _f32, _vp]),
    "xs_attn_fwd": (_int, [_vp, _vp, _vp, _vp, _int, _int, _int, _int, _f32, _vp]),
    "xs_attn_heads_fwd": (_int, [_vp, _vp, _vp, ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _f32, _vp]),
    "xs_relayout_a2a": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _vp]),
    "xs_attn_a2a_fwd_staged": (_int, [_vp, _vp, _vp, ctypes.POINTER(_vp), _vp, _vp, _vp, ctypes.POINTER(_vp),
                                      _int, _int, _int, _int, _int, _f32, _vp, _size, _vp]),
    "xs_attn_workspace_bytes": (_int, [_int, _int, _int, _int, ctypes.POINTER(_size)]),
    "xs_attn_fwd_balanced": (_int, [_vp, _vp, _vp, _int, ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _f32,
                                    _vp, _size, _vp]),
    "xs_attn_fwd_balanced_noalloc": (_int, [_vp, _vp, _vp, _int, ctypes.POINTER(_vp), _int, _int, _int, _int, _int,
                                            _f32, _vp]),
    "xs_attn_causal_fwd": (_int, [_vp, _vp, _vp, _int, ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _f32,
                                  _vp]),
    "xs_attn_varlen_fwd": (_int, [_vp, _vp, _vp, ctypes.POINTER(_int), _int, _int, _int, ctypes.POINTER(_vp), _int,
                                  _int, _int, _int, _f32, _vp]),
    "xs_attn_ulysses_fwd": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                   ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _f32, _vp, _size, _vp]),
    "xs_relayout_a2a_inverse": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _int, _int, _int, _int, _int,
                                       _vp]),
    "xs_attn_ulysses_rank_fwd": (_int, [_vp, _vp, _vp, ctypes.POINTER(_vp), _int, _int, _int, _int, _int, _int, _f32,
                                        _vp, _size, _vp]),
    "xs_burst_gap": (_int, [_vp, _size, _int, _size, _int, ctypes.c_longlong, ctypes.c_longlong, _vp, _vp]),
    "xs_attn_get_device_error": (_int, [_vp]),
    "xs_attn_get_device_error_info": (_int, [_vp, ctypes.POINTER(_int), _int]),
    "xs_attn_error_string": (ctypes.c_char_p, [_int]),
    "xs_attn_last_cuda_error": (_int, []),
    "xs_attn_version": (_int, []),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: the CUDA library has not been built "
            "(run `python -c 'import __graft_entry__ as g; g.build()'`); there is no fallback")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = _load()


class XsError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib.xs_attn_error_string(code).decode()
        if code == XS_ERR_CUDA:
            msg += f" (cudaError {lib.xs_attn_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


def _check(code: int, where: str) -> None:
    if code != XS_OK:
        raise XsError(code, where)


def _ptr_array(ptrs):
    arr = (_vp * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bshd(t, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
        raise TypeError(f"{name} must be a contiguous CUDA bfloat16 tensor [B,S,H,D]")
    return t


def xs_attn_a2a_fwd(q, k, v, out_ptrs, scale: float, stream=None) -> None:
    """Fused attention; writes P sequence shards ``out_ptrs[p]`` of shape [B,S/P,H,D]."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v")
    outs = [_bshd(o, "out") for o in out_ptrs]
    _check(lib.xs_attn_a2a_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr_array([o.data_ptr() for o in outs]),
                               B, S, H, D, len(outs), scale, _stream_handle(stream)), "xs_attn_a2a_fwd")


def xs_attn_fwd(q, k, v, out, scale: float, stream=None) -> None:
    """Same attention kernel, one contiguous [B,S,H,D] output."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v"), _bshd(out, "out")
    _check(lib.xs_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, D, scale,
                           _stream_handle(stream)), "xs_attn_fwd")


def xs_attn_heads_fwd(q, k, v, heads, scale: float, stream=None) -> None:
    """Same attention kernel, writing the P Ulysses head shards [B,S,H/P,D]."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v")
    hs = [_bshd(x, "heads") for x in heads]
    _check(lib.xs_attn_heads_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr_array([x.data_ptr() for x in hs]),
                                 B, S, H, D, len(hs), scale, _stream_handle(stream)), "xs_attn_heads_fwd")


def xs_relayout_a2a(heads, out_ptrs, stream=None) -> None:
    """Separate All-to-All re-layout: head shards [B,S,H/P,D] -> sequence shards [B,S/P,H,D]."""
    hs = [_bshd(x, "heads") for x in heads]
    outs = [_bshd(o, "out") for o in out_ptrs]
    P = len(hs)
    B, S, Hl, D = hs[0].shape
    _check(lib.xs_relayout_a2a(_ptr_array([x.data_ptr() for x in hs]), _ptr_array([o.data_ptr() for o in outs]),
                               B, S, Hl * P, D, P, _stream_handle(stream)), "xs_relayout_a2a")


def xs_attn_ulysses_fwd(q_shards, k_shards, v_shards, out_shards, scale: float, workspace=None,
                        stream=None) -> None:
    """The Ulysses attention step of P virtual ranks in one launch: inputs are the P sequence
    shards [B,S/P,H,D] of Q, K and V, outputs the P sequence shards [B,S/P,H,D] of O."""
    qs = [_bshd(x, "q_shards") for x in q_shards]
    ks = [_bshd(x, "k_shards") for x in k_shards]
    vs = [_bshd(x, "v_shards") for x in v_shards]
    os_ = [_bshd(x, "out_shards") for x in out_shards]
    P = len(qs)
    B, Sl, H, D = qs[0].shape
    wp, wn = _ws(workspace)
    _check(lib.xs_attn_ulysses_fwd(_ptr_array([x.data_ptr() for x in qs]), _ptr_array([x.data_ptr() for x in ks]),
                                   _ptr_array([x.data_ptr() for x in vs]), _ptr_array([x.data_ptr() for x in os_]),
                                   B, Sl * P, H, D, P, scale, wp, wn, _stream_handle(stream)), "xs_attn_ulysses_fwd")


def xs_attn_ulysses_rank_fwd(q_heads, k_heads, v_heads, out_shard_ptrs, H: int, rank: int, scale: float,
                             workspace=None, stream=None) -> None:
    """Attention of Ulysses rank ``rank`` over its head shard [B,S,H/P,D] (q, k, v), storing
    every output row straight into ``out_shard_ptrs[p]`` (device addresses of the P ranks'
    sequence shards [B,S/P,H,D], which may belong to other processes) at global head
    rank*H/P + j.  ``out_shard_ptrs``: ints (device pointers) or CUDA tensors."""
    B, S, Hl, D = _bshd(q_heads, "q_heads").shape
    _bshd(k_heads, "k_heads"), _bshd(v_heads, "v_heads")
    ptrs = [p if isinstance(p, int) else _bshd(p, "out_shards").data_ptr() for p in out_shard_ptrs]
    P = len(ptrs)
    wp, wn = _ws(workspace)
    _check(lib.xs_attn_ulysses_rank_fwd(q_heads.data_ptr(), k_heads.data_ptr(), v_heads.data_ptr(), _ptr_array(ptrs),
                                        B, S, H, D, P, rank, scale, wp, wn, _stream_handle(stream)),
           "xs_attn_ulysses_rank_fwd")


def xs_relayout_a2a_inverse(seq_shards, heads, stream=None) -> None:
    """Separate pre-attention All-to-All: sequence shards [B,S/P,H,D] -> head shards [B,S,H/P,D]."""
    ss = [_bshd(x, "seq_shards") for x in seq_shards]
    hs = [_bshd(x, "heads") for x in heads]
    P = len(ss)
    B, Sl, H, D = ss[0].shape
    _check(lib.xs_relayout_a2a_inverse(_ptr_array([x.data_ptr() for x in ss]), _ptr_array([x.data_ptr() for x in hs]),
                                       B, Sl * P, H, D, P, _stream_handle(stream)), "xs_relayout_a2a_inverse")


def xs_burst_gap(dst, producers: int, burst_bytes: int, bursts: int, gap_ns: int, stream=None, lead_ns: int = 0):
    """Run the Burst-Gap store microbenchmark into the CUDA tensor ``dst`` (any dtype, contiguous);
    returns the device int64 tensor [bursts, producers] of burst issue times in ns."""
    import torch
    if not dst.is_cuda or not dst.is_contiguous():
        raise TypeError("dst must be a contiguous CUDA tensor")
    times = torch.empty((bursts, producers), dtype=torch.int64, device=dst.device)
    _check(lib.xs_burst_gap(dst.data_ptr(), dst.numel() * dst.element_size(), producers, burst_bytes, bursts,
                            lead_ns, gap_ns, times.data_ptr(), _stream_handle(stream)), "xs_burst_gap")
    return times


def xs_attn_a2a_fwd_staged(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev, scale: float,
                           workspace=None, stream=None) -> None:
    """Host-resident variant: H2D copies, fused kernel and D2H copies of the shards, all on ``stream``.
    ``workspace``: a :class:`Workspace` (balanced schedule) or None (plain schedule)."""
    B, S, H, D = q_host.shape
    P = len(out_dev)
    wp, wn = _ws(workspace)
    _check(lib.xs_attn_a2a_fwd_staged(
        q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), _ptr_array([o.data_ptr() for o in out_host]),
        q_dev.data_ptr(), k_dev.data_ptr(), v_dev.data_ptr(), _ptr_array([o.data_ptr() for o in out_dev]),
        B, S, H, D, P, scale, wp, wn, _stream_handle(stream)), "xs_attn_a2a_fwd_staged")


def xs_attn_workspace_bytes(B: int, S: int, H: int, D: int) -> int:
    """Workspace bytes the balanced schedule needs for this shape on the current device (0: no split)."""
    n = _size(0)
    _check(lib.xs_attn_workspace_bytes(B, S, H, D, ctypes.byref(n)), "xs_attn_workspace_bytes")
    return n.value


class Workspace:
    """A zero-filled device workspace for :func:`xs_attn_fwd_balanced` (torch-allocated,
    256-byte aligned).  ``Workspace.for_shape(B, S, H, D)`` sizes it for one shape;
    ``None`` is returned there when the shape needs none."""

    def __init__(self, nbytes: int, device="cuda"):
        import torch
        self.nbytes = int(nbytes)
        self._buf = torch.zeros(self.nbytes + 256, dtype=torch.uint8, device=device)
        base = self._buf.data_ptr()
        self.ptr = (base + 255) & ~255

    @classmethod
    def for_shape(cls, B: int, S: int, H: int, D: int, device="cuda"):
        n = xs_attn_workspace_bytes(B, S, H, D)
        return cls(n, device) if n else None


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.ptr, workspace.nbytes


def xs_attn_fwd_balanced(q, k, v, layout: int, outs, scale: float, workspace, stream=None) -> None:
    """The attention kernel with the last partial wave of tiles balanced over all SMs.
    ``layout``: XS_LAYOUT_A2A (P sequence shards), XS_LAYOUT_CONTIGUOUS (one [B,S,H,D]
    tensor) or XS_LAYOUT_HEADS (P head shards); ``workspace``: a :class:`Workspace` or None."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v")
    os_ = [_bshd(o, "out") for o in outs]
    wp, wn = _ws(workspace)
    _check(lib.xs_attn_fwd_balanced(q.data_ptr(), k.data_ptr(), v.data_ptr(), layout,
                                    _ptr_array([o.data_ptr() for o in os_]), B, S, H, D, len(os_), scale, wp, wn,
                                    _stream_handle(stream)), "xs_attn_fwd_balanced")


def xs_attn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status code."""
    return lib.xs_attn_get_device_error(_stream_handle(stream))


def xs_attn_get_device_error_info(stream=None):
    """Synchronise the stream; return (status code, record of the first device error as a
    dict) and clear both (see include/xsattn.h for the fields)."""
    info = (_int * 8)()
    code = lib.xs_attn_get_device_error_info(_stream_handle(stream), info, 8)
    keys = ("kind", "cta", "warp", "lane", "site", "detail0", "detail1", "detail2")
    return code, dict(zip(keys, list(info)))


def xs_attn_error_string(code: int) -> str:
    return lib.xs_attn_error_string(code).decode()


def xs_attn_fwd_balanced_noalloc(q, k, v, layout: int, outs, scale: float, stream=None) -> None:
    """:func:`xs_attn_fwd_balanced` with the library's own scratch array as workspace (no
    allocation on the call path; calls that overlap in time race on the one array)."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v")
    os_ = [_bshd(o, "out") for o in outs]
    _check(lib.xs_attn_fwd_balanced_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), layout,
                                            _ptr_array([o.data_ptr() for o in os_]), B, S, H, D, len(os_), scale,
                                            _stream_handle(stream)), "xs_attn_fwd_balanced_noalloc")


def xs_attn_causal_fwd(q, k, v, layout: int, outs, scale: float, stream=None) -> None:
    """Causal attention (row s attends to keys 0 .. s) with the fused output layouts:
    ``layout`` XS_LAYOUT_A2A (P sequence shards), XS_LAYOUT_CONTIGUOUS (one [B,S,H,D]
    tensor) or XS_LAYOUT_HEADS (P head shards)."""
    B, S, H, D = _bshd(q, "q").shape
    _bshd(k, "k"), _bshd(v, "v")
    os_ = [_bshd(o, "out") for o in outs]
    _check(lib.xs_attn_causal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), layout,
                                  _ptr_array([o.data_ptr() for o in os_]), B, S, H, D, len(os_), scale,
                                  _stream_handle(stream)), "xs_attn_causal_fwd")


def _thd(t, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
        raise TypeError(f"{name} must be a contiguous CUDA bfloat16 tensor [T,H,D]")
    return t


def xs_attn_varlen_fwd(q, k, v, seqlens, layout: int, outs, scale: float, causal: bool = False,
                       stream=None) -> None:
    """Attention over packed variable-length sequences: ``q``, ``k``, ``v`` are
    [T, H, D] bf16 holding sequences of lengths ``seqlens`` (host integers) back to
    back; each row attends to its own sequence (``causal=True``: to its own
    sequence's keys up to its own position; run as one causal launch per
    sequence).
    ``layout`` XS_LAYOUT_A2A (P shards [T/P, H, D]), XS_LAYOUT_CONTIGUOUS (one
    [T, H, D] tensor) or XS_LAYOUT_HEADS (P head shards [T, H/P, D])."""
    T, H, D = _thd(q, "q").shape
    _thd(k, "k"), _thd(v, "v")
    os_ = [_thd(o, "out") for o in outs]
    lens = (ctypes.c_int * max(1, len(seqlens)))(*[int(n) for n in seqlens])
    _check(lib.xs_attn_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens, len(seqlens), int(bool(causal)),
                                  layout, _ptr_array([o.data_ptr() for o in os_]), T, H, D, len(os_), scale,
                                  _stream_handle(stream)), "xs_attn_varlen_fwd")


def attn_a2a(q, k, v, P: int, scale: float | None = None, stream=None, workspace=None):
    """Allocate the P output shards with torch and run the fused path; returns the list of shards.
    With a :class:`Workspace` the balanced schedule is used."""
    import torch
    B, S, H, D = q.shape
    if scale is None:
        scale = D ** -0.5
    outs = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16, device=q.device) for _ in range(P)]
    if workspace is None:
        xs_attn_a2a_fwd(q, k, v, outs, scale, stream)
    else:
        xs_attn_fwd_balanced(q, k, v, XS_LAYOUT_A2A, outs, scale, workspace, stream)
    return outs
