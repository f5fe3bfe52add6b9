"""The C ABI on the host: the library loads, exports every symbol the header
declares, and rejects every invalid argument with its documented code before
touching CUDA (these calls use fake, never-dereferenced pointer values)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def xs():
    from conftest import build_library
    build_library()
    import dit_attention_ulysses_gb300 as xs
    return xs


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "xsattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(xs_\w+)\s*\(", src)))


def test_exports_match_header(xs):
    declared = _declared_functions()
    assert "xs_attn_a2a_fwd" in declared and len(declared) >= 8
    for name in declared:
        assert hasattr(xs.lib, name), f"{name} declared but not exported"
    assert sorted(xs.EXPORTS) == declared


def test_error_strings(xs):
    default = xs.xs_attn_error_string(-999)
    assert "unknown" in default
    for code in range(0, -16, -1):
        s = xs.xs_attn_error_string(code)
        assert s and s != default
    assert xs.lib.xs_attn_version() >= 100


# fake device addresses, 16-byte aligned and far apart; never dereferenced
GB = 1 << 30
Q, K, V = 0x10_0000_0000, 0x20_0000_0000, 0x30_0000_0000
OUT0 = 0x40_0000_0000


def _outs(n, base=OUT0, step=GB):
    arr = (ctypes.c_void_p * max(1, n))()
    for i in range(n):
        arr[i] = base + i * step
    return arr


def _a2a(xs, q=Q, k=K, v=V, outs=None, B=1, S=256, H=2, D=64, P=2, scale=0.125):
    if outs is None:
        outs = _outs(P if 0 < P <= 16 else 1)
    return xs.lib.xs_attn_a2a_fwd(q, k, v, outs, B, S, H, D, P, scale, None)


def test_null_pointers(xs):
    assert _a2a(xs, q=None) == xs.XS_ERR_NULL
    assert _a2a(xs, v=None) == xs.XS_ERR_NULL
    assert xs.lib.xs_attn_a2a_fwd(Q, K, V, None, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_NULL
    outs = _outs(2)
    outs[1] = None
    assert _a2a(xs, outs=outs) == xs.XS_ERR_NULL
    assert xs.lib.xs_attn_fwd(Q, K, V, None, 1, 256, 2, 64, 0.1, None) == xs.XS_ERR_NULL
    assert xs.lib.xs_relayout_a2a(None, _outs(2), 1, 256, 2, 64, 2, None) == xs.XS_ERR_NULL


@pytest.mark.parametrize("B,S,H,P", [(0, 256, 2, 2), (1, 0, 2, 2), (1, 256, 0, 2), (1, 256, 2, 0), (-1, 256, 2, 2)])
def test_bad_shapes(xs, B, S, H, P):
    assert _a2a(xs, B=B, S=S, H=H, P=P) == xs.XS_ERR_SHAPE


@pytest.mark.parametrize("D", [0, 32, 96, 256, 65])
def test_bad_head_dim(xs, D):
    assert _a2a(xs, D=D) == xs.XS_ERR_HEAD_DIM


def test_too_many_ranks(xs):
    assert _a2a(xs, S=1024 * 17, H=17, P=17, outs=_outs(17)) == xs.XS_ERR_TOO_MANY_RANKS


@pytest.mark.parametrize("S,H,P", [(255, 2, 2), (256, 3, 2), (300, 12, 8)])
def test_divisibility(xs, S, H, P):
    assert _a2a(xs, S=S, H=H, P=P) == xs.XS_ERR_DIVISIBILITY


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), -0.5])
def test_bad_scale(xs, scale):
    assert _a2a(xs, scale=scale) == xs.XS_ERR_SCALE


def test_misaligned(xs):
    assert _a2a(xs, q=Q + 8) == xs.XS_ERR_ALIGNMENT
    assert _a2a(xs, outs=_outs(2, base=OUT0 + 2)) == xs.XS_ERR_ALIGNMENT


def test_overlap(xs):
    shard = 1 * 128 * 2 * 64 * 2  # bytes of one [1,128,2,64] shard
    assert _a2a(xs, outs=_outs(2, step=shard - 16)) == xs.XS_ERR_OVERLAP      # shards overlap
    assert _a2a(xs, outs=_outs(2, base=Q + 64)) == xs.XS_ERR_OVERLAP           # shard inside q
    assert _a2a(xs, outs=_outs(2, base=V - shard + 16)) == xs.XS_ERR_OVERLAP   # shard tail inside v
    # exactly adjacent is fine: validation passes, so the call reaches CUDA
    rc = _a2a(xs, outs=_outs(2, step=shard))
    assert rc not in (xs.XS_ERR_OVERLAP, xs.XS_ERR_NULL, xs.XS_ERR_ALIGNMENT, xs.XS_ERR_SHAPE)


def test_heads_and_relayout_validation(xs):
    lib = xs.lib
    assert lib.xs_attn_heads_fwd(Q, K, V, _outs(2), 1, 256, 3, 64, 2, 0.1, None) == xs.XS_ERR_DIVISIBILITY
    heads = _outs(2, base=0x50_0000_0000)
    assert lib.xs_relayout_a2a(heads, _outs(2), 1, 256, 2, 128, 2, None) not in (
        xs.XS_ERR_NULL, xs.XS_ERR_SHAPE, xs.XS_ERR_OVERLAP, xs.XS_ERR_ALIGNMENT)
    assert lib.xs_relayout_a2a(heads, _outs(2, base=0x50_0000_0000 + 4096), 1, 256, 2, 128, 2, None) == xs.XS_ERR_OVERLAP
    assert lib.xs_relayout_a2a(heads, _outs(2), 1, 256, 2, 48, 2, None) == xs.XS_ERR_HEAD_DIM


def test_staged_validation(xs):
    lib = xs.lib
    host = _outs(2, base=0x70_0000_0000)
    assert lib.xs_attn_a2a_fwd_staged(None, 1, 1, host, Q, K, V, _outs(2), 1, 256, 2, 64, 2, 0.1,
                                      None, 0, None) == xs.XS_ERR_NULL
    host3 = _outs(3, base=0x70_0000_0000)
    assert lib.xs_attn_a2a_fwd_staged(16, 16, 16, host3, Q, K, V, _outs(3), 1, 256, 2, 64, 3, 0.1,
                                      None, 0, None) == xs.XS_ERR_DIVISIBILITY
    # a workspace that overlaps an input is refused before anything runs
    assert lib.xs_attn_a2a_fwd_staged(16, 16, 16, host, Q, K, V, _outs(2), 1, 256, 2, 64, 2, 0.1,
                                      Q, 1 << 20, None) == xs.XS_ERR_OVERLAP


def test_balanced_validation(xs):
    lib = xs.lib
    WS = 0x60_0000_0000
    outs = _outs(2)
    # unknown layout
    assert lib.xs_attn_fwd_balanced(Q, K, V, 7, outs, 1, 256, 2, 64, 2, 0.1, WS, 1 << 20, None) == xs.XS_ERR_LAYOUT
    # layouts keep the checks of their plain entry points
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 3, 64, 2, 0.1, WS, 1 << 20, None) == \
        xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_HEADS, outs, 1, 255, 2, 64, 2, 0.1, WS, 1 << 20, None) == \
        xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_A2A, None, 1, 256, 2, 64, 2, 0.1, WS, 1 << 20, None) == \
        xs.XS_ERR_NULL
    # the workspace must be 256-byte aligned and disjoint from inputs and outputs
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 2, 64, 2, 0.1, WS + 16, 1 << 20,
                                    None) == xs.XS_ERR_ALIGNMENT
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 2, 64, 2, 0.1, K - 4096, 1 << 20,
                                    None) == xs.XS_ERR_OVERLAP
    ptrs = [outs[i] for i in range(2)]
    assert lib.xs_attn_fwd_balanced(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 2, 64, 2, 0.1, ptrs[1], 1 << 20,
                                    None) == xs.XS_ERR_OVERLAP


def test_causal_validation(xs):
    lib = xs.lib
    outs = _outs(2)
    A2A, CONT, HEADS = xs.XS_LAYOUT_A2A, xs.XS_LAYOUT_CONTIGUOUS, xs.XS_LAYOUT_HEADS
    assert lib.xs_attn_causal_fwd(Q, K, V, 7, outs, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_LAYOUT
    assert lib.xs_attn_causal_fwd(Q, K, V, A2A, None, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_NULL
    assert lib.xs_attn_causal_fwd(None, K, V, A2A, outs, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_NULL
    assert lib.xs_attn_causal_fwd(Q, K, V, A2A, outs, 1, 256, 3, 64, 2, 0.1, None) == xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_causal_fwd(Q, K, V, HEADS, outs, 1, 255, 2, 64, 2, 0.1, None) == xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_causal_fwd(Q, K, V, A2A, outs, 1, 256, 2, 96, 2, 0.1, None) == xs.XS_ERR_HEAD_DIM
    assert lib.xs_attn_causal_fwd(Q, K, V, A2A, outs, 0, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_SHAPE
    assert lib.xs_attn_causal_fwd(Q, K, V, A2A, outs, 1, 256, 2, 64, 2, float("nan"), None) == xs.XS_ERR_SCALE
    assert lib.xs_attn_causal_fwd(Q + 8, K, V, A2A, outs, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_ALIGNMENT
    assert lib.xs_attn_causal_fwd(Q, K, V, CONT, _outs(1, base=V + 4096), 1, 256, 2, 64, 1, 0.1, None) == \
        xs.XS_ERR_OVERLAP


def test_varlen_validation(xs):
    lib = xs.lib
    outs = _outs(2)
    A2A, CONT = xs.XS_LAYOUT_A2A, xs.XS_LAYOUT_CONTIGUOUS

    def call(lens, T=None, causal=0, layout=A2A, o=outs, H=2, D=64, P=2, q=Q, scale=0.1):
        arr = (ctypes.c_int * max(1, len(lens)))(*lens)
        T = sum(lens) if T is None else T
        return lib.xs_attn_varlen_fwd(q, K, V, arr, len(lens), causal, layout, o, T, H, D, P, scale, None)

    assert lib.xs_attn_varlen_fwd(Q, K, V, None, 1, 0, A2A, outs, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_NULL
    assert call([256], o=None) == xs.XS_ERR_NULL
    assert call([]) == xs.XS_ERR_SHAPE                          # no sequence
    assert call([1] * 1025, T=1026) == xs.XS_ERR_SHAPE          # too many sequences
    assert call([300, -44]) == xs.XS_ERR_SHAPE                  # negative length
    assert call([100, 156], T=250) == xs.XS_ERR_SHAPE           # lengths do not sum to T
    assert call([4097 * 128], layout=CONT, P=1) == xs.XS_ERR_SHAPE       # 4097 tiles
    assert call([8388609], layout=CONT, P=1) == xs.XS_ERR_SHAPE          # sequence too long
    assert call([0, 0]) == xs.XS_ERR_SHAPE                      # T = 0
    assert call([100, 156], layout=9) == xs.XS_ERR_LAYOUT
    assert call([100, 155]) == xs.XS_ERR_DIVISIBILITY           # T % P != 0 for the A2A shards
    assert call([100, 156], H=3) == xs.XS_ERR_DIVISIBILITY
    assert call([100, 156], D=96) == xs.XS_ERR_HEAD_DIM
    assert call([100, 156], q=Q + 8) == xs.XS_ERR_ALIGNMENT
    assert call([100, 156], scale=-1.0) == xs.XS_ERR_SCALE
    assert call([100, 156], layout=CONT, P=1, o=_outs(1, base=K + 64)) == xs.XS_ERR_OVERLAP
    # 1024 one-row sequences are 1024 tiles; with 2**21 + 1 heads the work units
    # (tiles x heads) would overflow an int although the dense-shape limits hold
    assert call([1] * 1024, layout=CONT, P=1, H=2 ** 21 + 1, D=64) == xs.XS_ERR_SHAPE
    # the causal form (one causal launch per sequence) takes the same host checks,
    # and a valid call gets as far as the non-causal one (no GPU here)
    assert call([100, 155], causal=1) == xs.XS_ERR_DIVISIBILITY
    assert call([100, 156], causal=1, D=96) == xs.XS_ERR_HEAD_DIM
    assert call([100, 156], causal=1, q=Q + 8) == xs.XS_ERR_ALIGNMENT
    assert call([100, 156], causal=1) == call([100, 156])
    assert call([256], causal=7, layout=CONT, P=1) == call([256], layout=CONT, P=1)


def test_workspace_query_validation(xs):
    import ctypes
    lib = xs.lib
    n = ctypes.c_size_t(0)
    assert lib.xs_attn_workspace_bytes(1, 256, 2, 64, None) == xs.XS_ERR_NULL
    assert lib.xs_attn_workspace_bytes(1, 256, 2, 48, ctypes.byref(n)) == xs.XS_ERR_HEAD_DIM
    assert lib.xs_attn_workspace_bytes(0, 256, 2, 64, ctypes.byref(n)) == xs.XS_ERR_SHAPE


def test_python_binding_rejects_cpu_tensors(xs):
    import torch
    q = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        xs.xs_attn_a2a_fwd(q, q, q, [q, q], 0.125)


def test_ulysses_and_inverse_relayout_validation(xs):
    lib = xs.lib
    qs, ks, vs = _outs(2, base=0x10_0000_0000), _outs(2, base=0x20_0000_0000), _outs(2, base=0x30_0000_0000)
    outs = _outs(2)
    # (S/P) % 128 != 0: a tile would straddle two input shards
    assert lib.xs_attn_ulysses_fwd(qs, ks, vs, outs, 1, 384, 2, 64, 2, 0.1, None, 0, None) == xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_ulysses_fwd(qs, ks, vs, outs, 1, 512, 3, 64, 2, 0.1, None, 0, None) == xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_ulysses_fwd(None, ks, vs, outs, 1, 512, 2, 64, 2, 0.1, None, 0, None) == xs.XS_ERR_NULL
    # an output shard inside an input shard
    assert lib.xs_attn_ulysses_fwd(qs, ks, vs, _outs(2, base=0x20_0000_0000 + 4096), 1, 512, 2, 64, 2, 0.1,
                                   None, 0, None) == xs.XS_ERR_OVERLAP
    # the workspace inside an output shard
    assert lib.xs_attn_ulysses_fwd(qs, ks, vs, outs, 1, 512, 2, 64, 2, 0.1, outs[0], 1 << 20, None) == \
        xs.XS_ERR_OVERLAP
    assert lib.xs_attn_ulysses_fwd(qs, ks, vs, outs, 1, 512, 2, 64, 2, 0.1, 0x60_0000_0010, 1 << 20, None) == \
        xs.XS_ERR_ALIGNMENT
    assert lib.xs_relayout_a2a_inverse(qs, outs, 1, 256, 3, 64, 2, None) == xs.XS_ERR_DIVISIBILITY
    assert lib.xs_relayout_a2a_inverse(qs, _outs(2, base=0x10_0000_0000 + 4096), 1, 256, 2, 64, 2, None) == \
        xs.XS_ERR_OVERLAP


def test_device_error_info_arguments_checked_before_any_cuda_call(xs):
    import ctypes
    info = (ctypes.c_int * 8)()
    assert xs.lib.xs_attn_get_device_error_info(None, info, 9) == xs.XS_ERR_NULL
    assert xs.lib.xs_attn_get_device_error_info(None, None, 1) == xs.XS_ERR_NULL
    assert xs.lib.xs_attn_get_device_error_info(None, info, -1) == xs.XS_ERR_NULL
