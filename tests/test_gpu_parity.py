"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small and ragged cases use the full oracle; the index-coded layout test is
compared bit for bit; the fused, contiguous and head-shard + re-layout paths
must agree bit for bit; guard regions and canaries check that every shard
element is written exactly inside its buffer.
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


def _oracle_shards(q, k, v, scale, P):
    """Oracle shards, plus sum_j w_j |v_j| in the same layout (for the rounding bound)."""
    import oracle
    return oracle.attention_a2a(q, k, v, scale, P), oracle.attention_a2a(q, k, abs_bits(v), scale, P)


def _run_fused(xs, q, k, v, scale, P):
    qd, kd, vd = (bits_to_torch(x) for x in (q, k, v))
    B, S, H, D = q.shape
    outs = [torch.full((B, S // P, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_a2a_fwd(qd, kd, vd, outs, scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == 0
    return outs


CASES = [
    # name, B, S, H, D, P  (several tiles, ragged tails, shard boundaries inside tiles)
    ("tiny", 1, 256, 2, 64, 2),
    ("two_units_d128", 1, 512, 2, 128, 2),
    ("ragged_1000", 2, 1000, 4, 128, 2),
    ("ragged_300_p3", 1, 300, 6, 64, 3),
    ("one_key", 1, 1, 2, 128, 1),
    ("five_keys", 2, 5, 1, 64, 1),
    ("s129", 1, 129, 2, 128, 1),
    ("s384_p8", 1, 384, 8, 128, 8),
    ("b3_h5", 3, 640, 5, 64, 5),
    # the most shards the ABI takes (16): 65-row shards, so every 128-row tile is
    # routed to two or three of them
    ("p16_sl65", 1, 1040, 16, 64, 16),
]


@pytest.mark.parametrize("name,B,S,H,D,P", CASES, ids=[c[0] for c in CASES])
def test_random_vs_oracle(xs, name, B, S, H, D, P):
    w = di.Workload(name, B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=S + H)
    q, k, v = di.random_qkv(w)
    ref, mass = _oracle_shards(q, k, v, w.scale, P)
    outs = _run_fused(xs, q, k, v, w.scale, P)
    got = np.stack([torch_to_f64(o) for o in outs])
    assert_close(got, ref, mass, name)


def test_tiny_workload_vs_oracle(xs):
    w = di.WORKLOADS["tiny"]
    q, k, v = di.random_qkv(w)
    ref, mass = _oracle_shards(q, k, v, w.scale, w.P)
    got = np.stack([torch_to_f64(o) for o in _run_fused(xs, q, k, v, w.scale, w.P)])
    assert got.shape == (2, 1, 128, 2, 64)
    assert_close(got, ref, mass, "tiny")


def test_outlier_channels_small(xs):
    w = di.Workload("outl", B=1, H=4, S=1024, D=128, P=4, scale=1 / math.sqrt(128), outliers=4)
    q, k, v = di.random_qkv(w)
    ref, mass = _oracle_shards(q, k, v, w.scale, w.P)
    got = np.stack([torch_to_f64(o) for o in _run_fused(xs, q, k, v, w.scale, w.P)])
    assert_close(got, ref, mass, "outliers")


@pytest.mark.parametrize("B,S,H,D,P", [(1, 256, 2, 64, 2), (2, 1000, 4, 128, 4), (1, 4608, 24, 128, 4),
                                       (1, 1040, 16, 64, 16), (2, 2048, 32, 128, 16)])
def test_layout_bit_exact(xs, B, S, H, D, P):
    q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
    outs = [torch.full((B, S // P, H, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_a2a_fwd(q, k, v, outs, scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == 0
    Sl = S // P
    for p in range(P):
        exp = di.layout_code_value_torch(B, S, H, D, s_offset=p * Sl, S_rows=Sl)
        assert torch.equal(outs[p].view(torch.int16), exp.view(torch.int16)), f"shard {p}"


def test_q_zero_gives_mean_of_v(xs):
    B, S, H, D, P = 1, 1000, 4, 128, 4
    w = di.Workload("z", B=B, H=H, S=S, D=D, P=P, scale=0.1)
    _, k, v = di.random_qkv(w)
    q = np.zeros_like(k)
    outs = _run_fused(xs, q, k, v, 0.1, P)
    got = np.concatenate([torch_to_f64(o) for o in outs], axis=1)
    mean = di.bf16_bits_to_f32(v).astype(np.float64).mean(axis=1, keepdims=True)
    # P is exactly 1 in bf16: only fp32 summation and the bf16 output rounding remain
    assert np.abs(got - mean).max() <= 2 ** -8 * np.abs(mean).max() + 1e-6


def test_scale_zero_gives_mean_of_v(xs):
    w = di.Workload("s0", B=1, H=2, S=300, D=64, P=2, scale=0.0)
    q, k, v = di.random_qkv(w)
    got = np.concatenate([torch_to_f64(o) for o in _run_fused(xs, q, k, v, 0.0, 2)], axis=1)
    mean = di.bf16_bits_to_f32(v).astype(np.float64).mean(axis=1, keepdims=True)
    assert np.abs(got - mean).max() <= 2 ** -8 * np.abs(mean).max() + 1e-6


@pytest.mark.parametrize("B,S,H,D,P", [(1, 1024, 8, 128, 4), (2, 600, 6, 64, 3), (1, 1040, 16, 64, 16),
                                       (2, 2048, 32, 128, 16)])
def test_fused_equals_contiguous_and_serial_path(xs, B, S, H, D, P):
    w = di.Workload("abl", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=7)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    fused = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_a2a_fwd(q, k, v, fused, w.scale)
    contig = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    xs.xs_attn_fwd(q, k, v, contig, w.scale)
    heads = [torch.empty((B, S, H // P, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_heads_fwd(q, k, v, heads, w.scale)
    serial = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_relayout_a2a(heads, serial)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == 0
    Sl = S // P
    for p in range(P):
        assert torch.equal(fused[p].view(torch.int16), contig[:, p * Sl:(p + 1) * Sl].view(torch.int16))
        assert torch.equal(fused[p].view(torch.int16), serial[p].view(torch.int16))
    Hl = H // P
    for r in range(P):
        assert torch.equal(heads[r].view(torch.int16), contig[:, :, r * Hl:(r + 1) * Hl].view(torch.int16))


def test_guards_and_canaries(xs):
    """Shards carved from one buffer with guard gaps: every shard element is
    overwritten (no NaN canary left) and no guard element changes."""
    B, S, H, D, P = 2, 700, 4, 128, 4
    w = di.Workload("g", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D))
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    shard = B * (S // P) * H * D
    guard = 4096
    pool = torch.empty(guard + P * (shard + guard), dtype=torch.bfloat16, device="cuda")
    pool.view(torch.int16).fill_(0x7FC1)   # a NaN payload the kernel never produces
    outs = [pool[guard + p * (shard + guard): guard + p * (shard + guard) + shard].view(B, S // P, H, D)
            for p in range(P)]
    xs.xs_attn_a2a_fwd(q, k, v, outs, w.scale)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == 0
    bits = pool.view(torch.int16)
    for p in range(P):
        lo = guard + p * (shard + guard)
        assert not (bits[lo:lo + shard] == 0x7FC1).any(), f"shard {p} has unwritten elements"
        assert bool((bits[lo - guard:lo] == 0x7FC1).all()), f"guard before shard {p} touched"
    assert bool((bits[-guard:] == 0x7FC1).all())


def test_deterministic(xs):
    w = di.Workload("d", B=1, H=4, S=2048, D=128, P=4, scale=1 / math.sqrt(128))
    q, k, v = di.random_qkv(w)
    a = _run_fused(xs, q, k, v, w.scale, 4)
    b = _run_fused(xs, q, k, v, w.scale, 4)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_staged_host_entry_matches_device_entry(xs):
    """The host-buffer entry pipelines head groups (min(H, 8) equal groups, the
    first and the last halved where they hold two heads or more: here, 12 heads,
    eight groups of one or two heads, the last one cut in two; copies of the next
    group in, kernel of this one, copies of the last one out, on three streams);
    without a workspace every group runs whole tiles, whose arithmetic is the
    whole-tensor kernel's, so the shards agree bit for bit.  Two calls back to
    back on a side stream, on the same device buffers with different host
    inputs: the second call's copies must wait for the first call's kernels."""
    w1 = di.Workload("st", B=1, H=12, S=1024, D=128, P=4, scale=1 / math.sqrt(128))
    w2 = di.Workload("st2", B=1, H=12, S=1024, D=128, P=4, scale=1 / math.sqrt(128), seed=9)
    pin = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    shape = (1, 256, 12, 128)
    qd, kd, vd = (torch.empty((1, 1024, 12, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out_d = [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    side = torch.cuda.Stream()
    outs, devs, keep = [], [], []
    for w in (w1, w2):
        qb, kb, vb = di.random_qkv(w)
        devs.append(_run_fused(xs, qb, kb, vb, w.scale, 4))
        out_h = [torch.full(shape, float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
        keep.append([pin(x) for x in (qb, kb, vb)])   # host inputs live until the stream is done
        xs.xs_attn_a2a_fwd_staged(*keep[-1], out_h, qd, kd, vd, out_d, w.scale, stream=side)
        outs.append(out_h)
    side.synchronize()
    assert xs.xs_attn_get_device_error(side) == xs.XS_OK
    for dev, out_h in zip(devs, outs):
        for a, b in zip(dev, out_h):
            assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16))


def test_non_default_stream(xs):
    w = di.Workload("ns", B=1, H=2, S=512, D=64, P=2, scale=0.125)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    ref = xs.attn_a2a(q, k, v, 2, 0.125)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = xs.attn_a2a(q, k, v, 2, 0.125)
    s.synchronize()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _scaled_keys_case(xs, key_rows, factor, S=512, H=2, D=128, P=2, seed=11):
    """Random inputs with a block of key rows scaled up, so that a later key block
    holds scores far above the running max (exercises the rescale paths)."""
    w = di.Workload("sk", B=1, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=seed)
    q, k, v = di.random_qkv(w)
    kf = di.bf16_bits_to_f32(k)
    kf[:, key_rows] *= factor
    k = di.f32_to_bf16_bits(kf)
    ref, mass = _oracle_shards(q, k, v, w.scale, P)
    got = np.stack([torch_to_f64(o) for o in _run_fused(xs, q, k, v, w.scale, P)])
    assert_close(got, ref, mass, f"scaled keys {key_rows} x{factor}")


def test_block_max_jump_first_half(xs):
    # first half of key block 1 scaled x4: its max exceeds the running max by more
    # than the lazy-rescale threshold, so O and l are rescaled
    _scaled_keys_case(xs, slice(128, 192), 4.0)


def test_block_max_jump_second_half(xs):
    # second half of key block 1 scaled x16: a very large jump, seen only by the
    # threads that own the second half of the keys
    _scaled_keys_case(xs, slice(192, 256), 16.0)


def test_block_max_jump_d64(xs):
    _scaled_keys_case(xs, slice(128, 192), 24.0, S=640, H=4, D=64, P=4, seed=3)


def test_growing_scores_every_block(xs):
    # every key block scaled a little more than the one before
    w = di.Workload("grow", B=1, H=2, S=1024, D=128, P=2, scale=1 / math.sqrt(128), seed=5)
    q, k, v = di.random_qkv(w)
    kf = di.bf16_bits_to_f32(k)
    for blk in range(8):
        kf[:, blk * 128:(blk + 1) * 128] *= 1.0 + 1.5 * blk
    k = di.f32_to_bf16_bits(kf)
    ref, mass = _oracle_shards(q, k, v, w.scale, 2)
    got = np.stack([torch_to_f64(o) for o in _run_fused(xs, q, k, v, w.scale, 2)])
    assert_close(got, ref, mass, "growing")
