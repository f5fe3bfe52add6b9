"""GPU parity of the whole Ulysses step in one launch (xs_attn_ulysses_fwd):
inputs are the P sequence shards of Q, K and V, outputs the P sequence shards
of O; the pre-attention exchange is fused into the TMA loads, the
post-attention one into the epilogue stores.  Also the separate pre-attention
re-layout kernel (xs_relayout_a2a_inverse) and the unfused Ulysses step built
from it.
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


def _split(bits, P):
    """[B,S,H,D] bits -> [P,B,S/P,H,D] sequence shards (rows [p*S/P, (p+1)*S/P))."""
    Sl = bits.shape[1] // P
    return np.stack([bits[:, p * Sl:(p + 1) * Sl] for p in range(P)])


def _shards_like(B, S, H, D, P, fill=float("nan")):
    return [torch.full((B, S // P, H, D), fill, dtype=torch.bfloat16, device="cuda") for _ in range(P)]


def _run_ulysses(xs, qs, ks, vs, scale, ws=None):
    P = len(qs)
    B, Sl, H, D = qs[0].shape
    outs = _shards_like(B, Sl * P, H, D, P)
    xs.xs_attn_ulysses_fwd(qs, ks, vs, outs, scale, ws)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    return outs


CASES = [
    # B, S, H, D, P: several tiles per shard, two shards; D = 64; eight shards of one tile
    (1, 1024, 4, 128, 2),
    (2, 768, 6, 64, 3),
    (1, 1024, 8, 128, 8),
]


@pytest.mark.parametrize("B,S,H,D,P", CASES, ids=[f"B{c[0]}_S{c[1]}_H{c[2]}_D{c[3]}_P{c[4]}" for c in CASES])
def test_ulysses_vs_oracle(xs, B, S, H, D, P):
    import oracle
    w = di.Workload("uly", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=S + P)
    q, k, v = di.random_qkv(w)
    sq, sk, sv = (_split(x, P) for x in (q, k, v))
    ref = oracle.ulysses_attention(sq, sk, sv, w.scale)
    mass = oracle.ulysses_attention(sq, sk, abs_bits(sv), w.scale)
    outs = _run_ulysses(xs, *[[bits_to_torch(x[p]) for p in range(P)] for x in (sq, sk, sv)], w.scale)
    assert_close(np.stack([torch_to_f64(o) for o in outs]), ref, mass, f"ulysses B={B} S={S} P={P}")


@pytest.mark.parametrize("B,S,H,D,P", CASES, ids=[f"B{c[0]}_S{c[1]}_H{c[2]}_D{c[3]}_P{c[4]}" for c in CASES])
def test_ulysses_bit_identical_to_fused_on_whole_tensors(xs, B, S, H, D, P):
    """Only the load addresses differ from xs_attn_a2a_fwd on the concatenated
    tensors, so the shards agree bit for bit (plain schedule)."""
    w = di.Workload("uly", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=5)
    q, k, v = di.random_qkv(w)
    Q, K, V = (bits_to_torch(x) for x in (q, k, v))
    ref = _shards_like(B, S, H, D, P)
    xs.xs_attn_a2a_fwd(Q, K, V, ref, w.scale)
    Sl = S // P
    sh = [[X[:, p * Sl:(p + 1) * Sl].contiguous() for p in range(P)] for X in (Q, K, V)]
    outs = _run_ulysses(xs, *sh, w.scale)
    for a, b in zip(outs, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ulysses_layout_bit_exact(xs):
    B, S, H, D, P = 2, 2048, 4, 128, 4
    q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
    Sl = S // P
    sh = [[X[:, p * Sl:(p + 1) * Sl].contiguous() for p in range(P)] for X in (q, k, v)]
    outs = _run_ulysses(xs, *sh, scale)
    for p in range(P):
        exp = di.layout_code_value_torch(B, S, H, D, s_offset=p * Sl, S_rows=Sl)
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"


def test_ulysses_full_size_video_small(xs):
    """Small video-DiT shape (4 shards of [1, 8192, 12, 128]) on the balanced
    schedule: layout bit-exact, then sampled rows against the oracle."""
    import oracle
    w = di.WORKLOADS["video_small"]
    P, Sl = w.P, w.S // w.P
    ws = xs.Workspace.for_shape(w.B, w.S, w.H, w.D)
    q, k, v, scale = di.layout_code_inputs_torch(w.B, w.S, w.H, w.D)
    sh = [[X[:, p * Sl:(p + 1) * Sl].contiguous() for p in range(P)] for X in (q, k, v)]
    del q, k, v
    outs = _run_ulysses(xs, *sh, scale, ws)
    for p in range(P):
        exp = di.layout_code_value_torch(w.B, w.S, w.H, w.D, s_offset=p * Sl, S_rows=Sl)
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"
    del sh, outs
    qb, kb, vb = di.random_qkv(w)
    sh = [[bits_to_torch(x[:, p * Sl:(p + 1) * Sl]) for p in range(P)] for x in (qb, kb, vb)]
    outs = _run_ulysses(xs, *sh, w.scale, ws)
    rb, rs = di.sample_rows(w, 48)
    ref = oracle.attention_rows(qb, kb, vb, w.scale, rb, rs)
    mass = oracle.attention_rows(qb, kb, abs_bits(vb), w.scale, rb, rs)
    got = np.stack([torch_to_f64(outs[int(s) // Sl][int(b), int(s) % Sl]) for b, s in zip(rb, rs)])
    assert_close(got, ref, mass, "ulysses video_small")


def test_relayout_inverse_bit_exact_and_round_trip(xs):
    """The separate pre-attention exchange: heads[r][b, s, j] = seq[s // Sl][b, s % Sl, r*Hl + j],
    checked element by element against NumPy slicing, and relayout_a2a undoes it."""
    B, S, H, D, P = 2, 384, 6, 64, 3
    x = di.random_qkv(di.Workload("r", B=B, H=H, S=S, D=D, P=P, scale=0.1, seed=9))[0]
    Sl, Hl = S // P, H // P
    seq = [bits_to_torch(x[:, p * Sl:(p + 1) * Sl]) for p in range(P)]
    heads = [torch.full((B, S, Hl, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_relayout_a2a_inverse(seq, heads)
    torch.cuda.synchronize()
    for r in range(P):
        want = x[:, :, r * Hl:(r + 1) * Hl]
        got = heads[r].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, want), f"rank {r}"
    back = _shards_like(B, S, H, D, P)
    xs.xs_relayout_a2a(heads, back)
    torch.cuda.synchronize()
    for p in range(P):
        assert torch.equal(back[p].view(torch.int16), seq[p].view(torch.int16))


def test_unfused_ulysses_step_matches_fused(xs):
    """Pre-attention re-layout of Q, K, V, attention of each rank on its head
    shard, post-attention re-layout: bit for bit the fused step."""
    B, S, H, D, P = 1, 1024, 8, 128, 4
    w = di.Workload("u2", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=13)
    bits = di.random_qkv(w)
    Sl, Hl = S // P, H // P
    sh = [[bits_to_torch(x[:, p * Sl:(p + 1) * Sl]) for p in range(P)] for x in bits]
    fused = _run_ulysses(xs, *sh, w.scale)
    heads = [[torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)] for _ in range(3)]
    for i in range(3):
        xs.xs_relayout_a2a_inverse(sh[i], heads[i])
    o_heads = [torch.empty((B, S, Hl, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    for r in range(P):
        xs.xs_attn_fwd(heads[0][r], heads[1][r], heads[2][r], o_heads[r], w.scale)
    serial = _shards_like(B, S, H, D, P)
    xs.xs_relayout_a2a(o_heads, serial)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    for a, b in zip(fused, serial):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ulysses_rejects_tiles_straddling_shards(xs):
    B, S, H, D, P = 1, 768, 4, 64, 4   # 192 rows per shard: not a multiple of 128
    q = [torch.zeros((B, S // P, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    outs = _shards_like(B, S, H, D, P)
    with pytest.raises(xs.XsError) as e:
        xs.xs_attn_ulysses_fwd(q, q, q, outs, 0.1)
    assert e.value.code == xs.XS_ERR_DIVISIBILITY


# ---- one rank's attention with the post-attention exchange in its epilogue
RANK_CASES = [
    # B, S, H, D, P
    (1, 1024, 8, 128, 4),
    (2, 1000, 4, 64, 2),      # shards of 500 rows: tiles straddle shard boundaries
    (1, 4608, 24, 128, 4),    # the image-DiT shape
]


def _rank_calls(xs, q, k, v, P, scale, ws=None):
    """P calls of xs_attn_ulysses_rank_fwd, rank r on heads [r*H/P, (r+1)*H/P)."""
    B, S, H, D = q.shape
    Hl = H // P
    outs = _shards_like(B, S, H, D, P)
    for r in range(P):
        sl = slice(r * Hl, (r + 1) * Hl)
        xs.xs_attn_ulysses_rank_fwd(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(), v[:, :, sl].contiguous(),
                                    outs, H, r, scale, ws)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    return outs


@pytest.mark.parametrize("B,S,H,D,P", RANK_CASES, ids=[f"B{c[0]}_S{c[1]}_H{c[2]}_D{c[3]}_P{c[4]}" for c in RANK_CASES])
def test_rank_entry_fills_shards_like_fused_kernel(xs, B, S, H, D, P):
    """Every rank stores its heads' rows into all P shards at head offset r*H/P;
    together the P calls give the fused kernel's shards bit for bit (a head's
    tiles do the same arithmetic whatever other heads the launch holds)."""
    w = di.Workload("rank", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=S + H)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    got = _rank_calls(xs, q, k, v, P, w.scale)
    ref = _shards_like(B, S, H, D, P)
    xs.xs_attn_a2a_fwd(q, k, v, ref, w.scale)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_rank_entry_layout_code_and_balanced_vs_oracle(xs):
    """Index-coded inputs: every output row is its own V row at its global head;
    and random inputs with the balanced schedule (workspace sized for H/P heads)
    against the oracle's whole path."""
    import oracle
    B, S, H, D, P = 1, 4096, 10, 128, 2
    q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
    outs = _rank_calls(xs, q, k, v, P, scale)
    Sl = S // P
    for p in range(P):
        exp = di.layout_code_value_torch(B, S, H, D, s_offset=p * Sl, S_rows=Sl)
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"
    w = di.Workload("rankbal", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=5)
    qb, kb, vb = di.random_qkv(w)
    need = xs.xs_attn_workspace_bytes(B, S, H // P, D)
    assert need > 0, "5 heads of 32 tiles leave 8 tiles to split on 152 SMs"
    ws = xs.Workspace(need)
    outs = _rank_calls(xs, *(bits_to_torch(x) for x in (qb, kb, vb)), P, w.scale, ws)
    ref = oracle.attention_a2a(qb, kb, vb, w.scale, P)
    mass = oracle.attention_a2a(qb, kb, abs_bits(vb), w.scale, P)
    assert_close(np.stack([torch_to_f64(o) for o in outs]), ref, mass, "rank entry, balanced")


def test_rank_entry_rejects_bad_rank(xs):
    q = torch.zeros((1, 256, 1, 64), dtype=torch.bfloat16, device="cuda")
    outs = _shards_like(1, 256, 2, 64, 2)
    with pytest.raises(xs.XsError) as e:
        xs.xs_attn_ulysses_rank_fwd(q, q, q, outs, 2, 2, 0.1)
    assert e.value.code == xs.XS_ERR_SHAPE
