"""GPU parity of causal attention (xs_attn_causal_fwd): query row s attends to
keys 0 .. s.  Tiles read key blocks 0 .. t only (t = the query tile) and the
diagonal block is masked per row.  Tiles run in one of two orders chosen on the
host (longest first with the heads side by side, or head-major where that
balances as well); both are exercised.

Checked against the fp64 oracle's causal entries (element by element at
sizes the oracle finishes in seconds, spanning several tiles, more than one
wave of tiles and ragged sequence tails; sampled rows at the image-DiT and
small video-DiT shapes), bit for bit on the index-coded layout inputs,
the three output layouts against each other, guard regions around the
output shards, the closed form for Q = 0 (prefix means of V), and the last
row of every head against the bidirectional kernel (the same keys and the same
arithmetic, so bit for bit).
"""
import math

import numpy as np
import pytest

import dit_inputs as di
from _parity import abs_bits, assert_close, bits_to_torch, torch_to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def xs():
    from conftest import build_library
    build_library()
    import dit_attention_ulysses_gb300 as xs
    assert torch.cuda.is_available()
    return xs


def _shards(B, S, H, D, P, fill=float("nan")):
    return [torch.full((B, S // P, H, D), fill, dtype=torch.bfloat16, device="cuda") for _ in range(P)]


def _causal(xs, q, k, v, P, scale, layout=None):
    B, S, H, D = q.shape
    if layout is None:
        layout = xs.XS_LAYOUT_A2A
    if layout == xs.XS_LAYOUT_CONTIGUOUS:
        outs = [torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")]
    elif layout == xs.XS_LAYOUT_HEADS:
        outs = [torch.full((B, S, H // P, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    else:
        outs = _shards(B, S, H, D, P)
    xs.xs_attn_causal_fwd(q, k, v, layout, outs, scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    return outs


CASES = [
    # B, S, H, D, P
    (1, 1024, 2, 128, 2),    # 8 query tiles per head, 1 .. 8 key blocks
    (1, 4000, 5, 128, 5),    # ragged tail (4000 = 31*128 + 32); 160 tiles: more than one wave, snake order
    (2, 300, 2, 64, 2),      # D = 64, ragged, three tiles
    (3, 2176, 4, 64, 4),     # D = 64, 17 tiles per head
    (1, 128, 1, 128, 1),     # one tile: only the diagonal block
    (1, 1, 1, 64, 1),        # one row, one key
]


@pytest.mark.parametrize("B,S,H,D,P", CASES, ids=[f"B{c[0]}_S{c[1]}_H{c[2]}_D{c[3]}_P{c[4]}" for c in CASES])
def test_causal_vs_oracle(xs, B, S, H, D, P):
    import oracle
    w = di.Workload("causal", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=S + D)
    q, k, v = di.random_qkv(w)
    ref = oracle.attention_a2a(q, k, v, w.scale, P, causal=True)
    mass = oracle.attention_a2a(q, k, abs_bits(v), w.scale, P, causal=True)
    outs = _causal(xs, *(bits_to_torch(x) for x in (q, k, v)), P, w.scale)
    assert_close(np.stack([torch_to_f64(o) for o in outs]), ref, mass, f"causal B={B} S={S} H={H} D={D} P={P}")


def test_causal_layouts_bit_identical(xs):
    """A2A shards, the contiguous tensor and head shards hold the same values."""
    B, S, H, D, P = 1, 4000, 5, 128, 5
    w = di.Workload("lay", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=3)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    full = _causal(xs, q, k, v, 1, w.scale, xs.XS_LAYOUT_CONTIGUOUS)[0]
    a2a = _causal(xs, q, k, v, P, w.scale, xs.XS_LAYOUT_A2A)
    heads = _causal(xs, q, k, v, P, w.scale, xs.XS_LAYOUT_HEADS)
    Sl, Hl = S // P, H // P
    for p in range(P):
        assert torch.equal(a2a[p].view(torch.int16), full[:, p * Sl:(p + 1) * Sl].view(torch.int16))
        assert torch.equal(heads[p].view(torch.int16), full[:, :, p * Hl:(p + 1) * Hl].view(torch.int16))


def test_causal_guard_regions_and_every_element_written(xs):
    """The shards sit between guard regions of one buffer, all holding a NaN
    pattern: afterwards no guard element has changed and no shard element still
    holds the pattern (every output element was written; outputs are finite)."""
    B, S, H, D, P = 2, 1000, 4, 64, 4
    w = di.Workload("guard", B=B, H=H, S=S, D=D, P=P, scale=0.125, seed=11)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    n, guard = B * (S // P) * H * D, 4096
    PATTERN = 0x7FC1
    buf = torch.full((guard + P * (n + guard),), PATTERN, dtype=torch.int16, device="cuda")
    outs = [buf[guard + p * (n + guard): guard + p * (n + guard) + n].view(torch.bfloat16).view(B, S // P, H, D)
            for p in range(P)]
    xs.xs_attn_causal_fwd(q, k, v, xs.XS_LAYOUT_A2A, outs, w.scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    mask = torch.ones_like(buf, dtype=torch.bool)
    for p in range(P):
        mask[guard + p * (n + guard): guard + p * (n + guard) + n] = False
    assert torch.all(buf[mask] == PATTERN), "a store landed outside the output shards"
    assert not torch.any(buf[~mask] == PATTERN), "an output element was not written"
    assert all(torch.isfinite(o.float()).all() for o in outs)


def test_causal_q_zero_gives_prefix_means(xs):
    """Q = 0: every unmasked score is 0, every probability exactly 1, and row s
    is the mean of V[0 .. s] (fp32 sums of bf16 products, rounded to bf16)."""
    B, S, H, D = 1, 1000, 3, 128
    w = di.Workload("q0", B=B, H=H, S=S, D=D, P=1, scale=0.1, seed=21)
    _, k, v = di.random_qkv(w)
    q = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    out = _causal(xs, q, bits_to_torch(k), bits_to_torch(v), 1, w.scale, xs.XS_LAYOUT_CONTIGUOUS)[0]
    vf = di.bf16_bits_to_f32(v).astype(np.float64)
    ref = np.cumsum(vf, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    got = torch_to_f64(out)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
    # the first row copies V[0] exactly
    np.testing.assert_array_equal(got[:, 0], vf[:, 0])


@pytest.mark.parametrize("S", [4608, 4000])
def test_causal_last_row_equals_bidirectional(xs, S):
    """Row S-1 attends to every key in both kernels, through the same blocks in
    the same order with the same masks: bit-identical results."""
    B, H, D = 1, 24, 128
    w = di.Workload("last", B=B, H=H, S=S, D=D, P=1, scale=1 / math.sqrt(D), seed=7)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    causal = _causal(xs, q, k, v, 1, w.scale, xs.XS_LAYOUT_CONTIGUOUS)[0]
    full = torch.full_like(causal, float("nan"))
    xs.xs_attn_fwd(q, k, v, full, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(causal[:, -1].view(torch.int16), full[:, -1].view(torch.int16))
    assert not torch.equal(causal[:, 0].view(torch.int16), full[:, 0].view(torch.int16))


@pytest.mark.parametrize("B,S,H,D,P", [(1, 4608, 24, 128, 4), (1, 4000, 5, 128, 5), (2, 512, 4, 64, 2),
                                       (1, 75776, 40, 128, 8), (1, 1040, 16, 64, 16)],
                         ids=["image", "ragged_two_waves", "d64", "video_large", "p16_sl65"])
def test_causal_layout_code_bit_exact(xs, B, S, H, D, P):
    """Index-coded inputs: the own key dominates every other by a weight ratio
    below fp32 resolution and lies inside the causal window, so every output
    row is its own V row exactly, in the owning shard at the right head.  The
    image shape runs the longest-first tile order, the others the head-major
    one (the large video-DiT shape at full size)."""
    q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
    outs = _causal(xs, q, k, v, P, scale)
    Sl = S // P
    for p in range(P):
        exp = di.layout_code_value_torch(B, S, H, D, s_offset=p * Sl, S_rows=Sl)
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"


@pytest.mark.parametrize("name,n_rows", [("image", 64), ("video_small", 48)])
def test_causal_full_size_sampled_rows(xs, name, n_rows):
    """The image-DiT and small video-DiT shapes: sampled rows (the first and last
    row of every shard among them, plus the first rows of the sequence, whose
    windows are shortest) against the oracle."""
    import oracle
    w = di.WORKLOADS[name]
    qb, kb, vb = di.random_qkv(w)
    outs = _causal(xs, *(bits_to_torch(x) for x in (qb, kb, vb)), w.P, w.scale)
    rb, rs = di.sample_rows(w, n_rows)
    rb = np.concatenate([rb, np.zeros(4, dtype=np.int64)])
    rs = np.concatenate([rs, np.array([1, 2, 127, 128], dtype=np.int64)])
    ref = oracle.attention_rows(qb, kb, vb, w.scale, rb, rs, causal=True)
    mass = oracle.attention_rows(qb, kb, abs_bits(vb), w.scale, rb, rs, causal=True)
    Sl = w.S // w.P
    got = np.stack([torch_to_f64(outs[int(s) // Sl][int(b), int(s) % Sl]) for b, s in zip(rb, rs)])
    assert_close(got, ref, mass, f"causal {name}")
