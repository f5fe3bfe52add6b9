"""GPU parity of attention over packed variable-length sequences
(xs_attn_varlen_fwd): sequences of given lengths lie back to back in one
[T, H, D] tensor per operand and every row attends to its own sequence (causal:
up to its own position; that form runs as one causal launch per sequence).

Checked against the oracle's attention_varlen, both forms (element by element
on mixes of lengths that are below, at and above one 128-row tile, with empty
sequences), bit for bit against the dense kernels when all lengths are equal
(the packed tensor is then the [B, S, H, D] tensor), bit for bit on index-coded
inputs (including the large video shape's 75,776 tokens as four sequences), the
three output layouts against each other, guard regions around the shards, the
closed forms for Q = 0 (sequence means; causal: prefix means), and sampled rows
of the largest call the table admits (1024 sequences, 4096 tiles).
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


def _packed_inputs(seqlens, H, D, seed):
    T = sum(seqlens)
    w = di.Workload("varlen", B=1, H=H, S=T, D=D, P=1, scale=1 / math.sqrt(D), seed=seed)
    return di.random_qkv(w), w.scale


def _run(xs, q, k, v, seqlens, layout, P, scale, causal=False):
    T, H, D = q.shape
    if layout == xs.XS_LAYOUT_CONTIGUOUS:
        outs = [torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")]
    elif layout == xs.XS_LAYOUT_HEADS:
        outs = [torch.full((T, H // P, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    else:
        outs = [torch.full((T // P, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_varlen_fwd(q, k, v, seqlens, layout, outs, scale, causal=causal)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    return outs


def _dev(bits):
    return bits_to_torch(bits[0])   # [1, T, H, D] bits -> [T, H, D] device tensor


CASES = [
    # seqlens, H, D, P (A2A shards of the packed rows)
    ([500, 12, 700, 300], 4, 128, 4),            # T = 1512; tiles of 1 .. 6 blocks, a 12-row sequence
    ([1, 127, 128, 129, 300, 1000, 3], 2, 128, 2),  # lengths around one tile; T = 1688
    ([33, 1, 250, 160], 2, 64, 2),               # D = 64; T = 444
    ([0, 640, 0, 0, 384], 3, 128, 1),            # empty sequences
]


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
@pytest.mark.parametrize("seqlens,H,D,P", CASES, ids=["mix1", "around_tile", "d64", "empty_seqs"])
def test_varlen_vs_oracle(xs, seqlens, H, D, P, causal):
    import oracle
    (q, k, v), scale = _packed_inputs(seqlens, H, D, seed=len(seqlens) + D)
    ref = oracle.attention_varlen(q, k, v, seqlens, scale, causal=causal)[0]
    mass = oracle.attention_varlen(q, k, abs_bits(v), seqlens, scale, causal=causal)[0]
    outs = _run(xs, _dev(q), _dev(k), _dev(v), seqlens, xs.XS_LAYOUT_A2A, P, scale, causal=causal)
    got = np.concatenate([torch_to_f64(o) for o in outs], axis=0)   # shards hold consecutive packed rows
    assert_close(got, ref, mass, f"varlen {seqlens} causal={causal}")


@pytest.mark.parametrize("B,S,H,D", [(3, 1000, 4, 128), (2, 2048, 2, 64)])
def test_varlen_equal_lengths_bit_identical_to_dense(xs, B, S, H, D):
    """Equal lengths: the packed tensor is the [B, S, H, D] tensor, every tile
    does the same arithmetic as in the dense kernel (keys past a sequence are
    masked in both; padding rows are not stored), so the outputs agree bit for bit."""
    w = di.Workload("eq", B=B, H=H, S=S, D=D, P=1, scale=1 / math.sqrt(D), seed=B * S)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    dense = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    xs.xs_attn_fwd(q, k, v, dense, w.scale)
    packed = _run(xs, *(x.view(B * S, H, D) for x in (q, k, v)), [S] * B, xs.XS_LAYOUT_CONTIGUOUS, 1, w.scale)[0]
    assert torch.equal(packed.view(torch.int16), dense.view(B * S, H, D).view(torch.int16))


@pytest.mark.parametrize("B,S,H,D", [(3, 1000, 4, 128), (2, 2048, 2, 64)])
def test_varlen_causal_equal_lengths_bit_identical_to_dense_causal(xs, B, S, H, D):
    """Equal lengths: each sequence's causal launch does the dense causal kernel's
    arithmetic for that batch entry, so the outputs agree bit for bit."""
    w = di.Workload("eqc", B=B, H=H, S=S, D=D, P=1, scale=1 / math.sqrt(D), seed=B * S + 1)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    dense = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    xs.xs_attn_causal_fwd(q, k, v, xs.XS_LAYOUT_CONTIGUOUS, [dense], w.scale)
    packed = _run(xs, *(x.view(B * S, H, D) for x in (q, k, v)), [S] * B, xs.XS_LAYOUT_CONTIGUOUS, 1, w.scale,
                  causal=True)[0]
    assert torch.equal(packed.view(torch.int16), dense.view(B * S, H, D).view(torch.int16))


def test_varlen_layouts_bit_identical(xs):
    seqlens, H, D, P = [500, 12, 700, 300], 4, 128, 4
    (q, k, v), scale = _packed_inputs(seqlens, H, D, seed=5)
    q, k, v = _dev(q), _dev(k), _dev(v)
    full = _run(xs, q, k, v, seqlens, xs.XS_LAYOUT_CONTIGUOUS, 1, scale)[0]
    a2a = _run(xs, q, k, v, seqlens, xs.XS_LAYOUT_A2A, P, scale)
    heads = _run(xs, q, k, v, seqlens, xs.XS_LAYOUT_HEADS, P, scale)
    T, Tl, Hl = sum(seqlens), sum(seqlens) // P, H // P
    for p in range(P):
        assert torch.equal(a2a[p].view(torch.int16), full[p * Tl:(p + 1) * Tl].view(torch.int16))
        assert torch.equal(heads[p].view(torch.int16), full[:, p * Hl:(p + 1) * Hl].view(torch.int16))


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
@pytest.mark.parametrize("seqlens,H,D,P", [([1000, 1, 129, 0, 918], 8, 128, 4),
                                           ([27916, 12272, 30881, 4707], 40, 128, 8),
                                           ([500, 12, 700, 324], 16, 64, 16)],
                         ids=["mix", "video_large_tokens", "p16_sl96"])
def test_varlen_layout_code_bit_exact(xs, seqlens, H, D, P, causal):
    """Index-coded inputs over the packed rows: each row's own key dominates
    every other key of its sequence, so every output row is its own V row.  The
    second case packs the large video-DiT shape's 75776 tokens as the bench's
    seeded mix of four sequences."""
    T = sum(seqlens)
    q, k, v, scale = di.layout_code_inputs_torch(1, T, H, D)
    outs = _run(xs, q[0], k[0], v[0], seqlens, xs.XS_LAYOUT_A2A, P, scale, causal=causal)
    Tl = T // P
    for p in range(P):
        exp = di.layout_code_value_torch(1, T, H, D, s_offset=p * Tl, S_rows=Tl)[0]
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_varlen_guard_regions_and_every_element_written(xs, causal):
    seqlens, H, D, P = [0, 300, 5, 0, 207], 4, 64, 2
    T = sum(seqlens)
    (q, k, v), scale = _packed_inputs(seqlens, H, D, seed=8)
    n, guard, PATTERN = (T // P) * H * D, 4096, 0x7FC1
    buf = torch.full((guard + P * (n + guard),), PATTERN, dtype=torch.int16, device="cuda")
    outs = [buf[guard + p * (n + guard): guard + p * (n + guard) + n].view(torch.bfloat16).view(T // P, H, D)
            for p in range(P)]
    xs.xs_attn_varlen_fwd(_dev(q), _dev(k), _dev(v), seqlens, xs.XS_LAYOUT_A2A, outs, scale, causal=causal)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    mask = torch.ones_like(buf, dtype=torch.bool)
    for p in range(P):
        mask[guard + p * (n + guard): guard + p * (n + guard) + n] = False
    assert torch.all(buf[mask] == PATTERN), "a store landed outside the output shards"
    assert not torch.any(buf[~mask] == PATTERN), "an output element was not written"


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_varlen_q_zero_gives_sequence_means(xs, causal):
    seqlens, H, D = [1, 200, 57, 130], 2, 128
    T = sum(seqlens)
    (_, k, v), scale = _packed_inputs(seqlens, H, D, seed=9)
    q = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    got = torch_to_f64(_run(xs, q, _dev(k), _dev(v), seqlens, xs.XS_LAYOUT_CONTIGUOUS, 1, scale, causal=causal)[0])
    vf = di.bf16_bits_to_f32(v[0]).astype(np.float64)
    start = 0
    for n in seqlens:
        seg = vf[start:start + n]
        if causal:   # row s: the mean of the sequence's rows 0 .. s
            ref = np.cumsum(seg, axis=0) / np.arange(1, n + 1)[:, None, None]
        else:
            ref = np.broadcast_to(seg.mean(axis=0, keepdims=True), seg.shape)
        bound = 2.0 ** -8 * np.abs(ref) + 1e-5
        assert np.all(np.abs(got[start:start + n] - ref) <= bound)
        start += n


def test_varlen_largest_table_sampled_rows(xs):
    """1024 sequences of 512 rows (4096 tiles, the table's limits): sampled rows
    against the oracle run on their own sequence."""
    import oracle
    n_seqs, L, H, D = 1024, 512, 1, 64
    seqlens = [L] * n_seqs
    (q, k, v), scale = _packed_inputs(seqlens, H, D, seed=10)
    out = _run(xs, _dev(q), _dev(k), _dev(v), seqlens, xs.XS_LAYOUT_CONTIGUOUS, 1, scale)[0]
    rng = np.random.default_rng(3)
    for seq in sorted(set([0, n_seqs - 1] + list(rng.integers(0, n_seqs, 6)))):
        sl = slice(seq * L, (seq + 1) * L)
        rows = np.array([0, 1, 127, 128, 300, L - 1], dtype=np.int64)
        zb = np.zeros_like(rows)
        ref = oracle.attention_rows(q[:, sl], k[:, sl], v[:, sl], scale, zb, rows)
        mass = oracle.attention_rows(q[:, sl], k[:, sl], abs_bits(v[:, sl]), scale, zb, rows)
        got = torch_to_f64(out[seq * L + torch.from_numpy(rows).cuda()])
        assert_close(got, ref, mass, f"sequence {seq}")


def test_varlen_rejects_bad_lengths(xs):
    q = torch.zeros((256, 2, 64), dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty((128, 2, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for causal in (False, True):
        with pytest.raises(xs.XsError) as e:
            xs.xs_attn_varlen_fwd(q, q, q, [100, 100], xs.XS_LAYOUT_A2A, outs, 0.1, causal=causal)
        assert e.value.code == xs.XS_ERR_SHAPE
