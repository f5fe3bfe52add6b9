"""The allocation-free entry point (xs_attn_fwd_balanced_noalloc) against the
entry point that takes a caller workspace (xs_attn_fwd_balanced).

Some callers cannot allocate device memory on their call path (a serving loop
that reserves all memory at start-up, where cudaMalloc may fail and cudaFree
would synchronise the device); the allocation-free entry point runs the
balanced schedule on the library's own scratch array instead.  The GPU tests
call it back to back on two shapes whose tiles are split (so the scratch array
is used) and whose per-CTA layouts differ (D = 64 on 152 CTAs, D = 128 on 128
CTAs), then on the first shape again, and compare every result bit for bit with
the workspace entry point on the same inputs.  Each call therefore starts on
scratch contents left by a call of the other shape.  This file sorts last, so a
run that stops at its first failure has run every other test before it."""
import math

import pytest

import dit_inputs as di
from _parity import bits_to_torch

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def xs():
    from conftest import build_library
    build_library()
    import dit_attention_ulysses_gb300 as xs
    return xs


def test_noalloc_checks_arguments_before_any_cuda_call(xs):
    """Runs without a GPU: invalid calls are refused on the host (fake pointers)."""
    import ctypes
    Q, K, V = 0x10_0000_0000, 0x20_0000_0000, 0x30_0000_0000
    outs = (ctypes.c_void_p * 2)(0x40_0000_0000, 0x40_4000_0000)
    lib = xs.lib
    assert lib.xs_attn_fwd_balanced_noalloc(Q, K, V, 7, outs, 1, 256, 2, 64, 2, 0.1, None) == xs.XS_ERR_LAYOUT
    assert lib.xs_attn_fwd_balanced_noalloc(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 3, 64, 2, 0.1, None) == \
        xs.XS_ERR_DIVISIBILITY
    assert lib.xs_attn_fwd_balanced_noalloc(Q, K, V, xs.XS_LAYOUT_A2A, None, 1, 256, 2, 64, 2, 0.1, None) == \
        xs.XS_ERR_NULL
    assert lib.xs_attn_fwd_balanced_noalloc(Q, K, V, xs.XS_LAYOUT_A2A, outs, 1, 256, 2, 64, 2, -1.0, None) == \
        xs.XS_ERR_SCALE


# (S, D, P, H): on a 152-SM GB300 the first splits its 192 tiles' last 40 over
# 152 CTAs, the second its 32 tiles over 128 CTAs
SHAPES = [(4096, 64, 2, 6), (4096, 128, 1, 1)]


def _call_both(xs, S, D, P, H, seed, ws):
    B = 1
    w = di.Workload("na", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=seed)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    ref = [torch.full((B, S // P, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    got = [torch.full((B, S // P, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, ref, w.scale, ws)
    xs.xs_attn_fwd_balanced_noalloc(q, k, v, xs.XS_LAYOUT_A2A, got, w.scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_across_shapes(xs):
    wss = []
    for S, D, P, H in SHAPES:
        need = xs.xs_attn_workspace_bytes(1, S, H, D)
        assert 0 < need <= 11 << 20, "the shape must split tiles and fit the scratch array"
        wss.append(xs.Workspace(need))
    for shape, seed in ((0, 21), (0, 22), (1, 23), (0, 24), (1, 25)):
        S, D, P, H = SHAPES[shape]
        _call_both(xs, S, D, P, H, seed, wss[shape])


@pytest.mark.gpu
def test_noalloc_argument_checks(xs):
    q = torch.zeros((1, 256, 2, 64), dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((1, 128, 2, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(xs.XsError) as e:
        xs.xs_attn_fwd_balanced_noalloc(q, q, q, 9, outs, 0.1)
    assert e.value.code == xs.XS_ERR_LAYOUT
    with pytest.raises(xs.XsError) as e:
        xs.xs_attn_fwd_balanced_noalloc(q, q, q, xs.XS_LAYOUT_A2A, outs, float("nan"))
    assert e.value.code == xs.XS_ERR_SCALE
