"""GPU parity of the balanced schedule (xs_attn_fwd_balanced): the tiles left
over after the whole waves are divided over the SMs by key blocks, and tiles
cut among CTAs are merged inside the kernel through the workspace.

The shapes split tiles on a 152-SM GB300 (each test asserts that they do on the
device at hand): into two pieces, into three, with a ragged key tail, at D = 64.
The full-size case also compares rows of every split tile, whose positions are
recomputed here from the schedule's definition.
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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


from _schedule import split_tiles  # noqa: E402


# (S, D, P, B, H) on 152 SMs: tiles cut in four (S=4096, H=5), in two or three
# (H=7), a ragged key tail with P=5 (S=4000), D = 64 (S=4096, H=6)
SHAPES = [
    (4096, 128, 1, 1, 5),
    (4096, 128, 1, 1, 7),
    (4000, 128, 5, 1, 5),
    (4096, 64, 2, 1, 6),
]


def _check_splits(B, S, H):
    n = (S + 127) // 128
    sp = split_tiles(B * H * n, n, _sms())
    assert sp, f"B={B} S={S} H={H} must split tiles on {_sms()} SMs"
    return sp


def _shards(B, S, H, D, P, fill=float("nan")):
    return [torch.full((B, S // P, H, D), fill, dtype=torch.bfloat16, device="cuda") for _ in range(P)]


def _run(xs, q, k, v, scale, P, ws, layout=None):
    B, S, H, D = q.shape
    layout = xs.XS_LAYOUT_A2A if layout is None else layout
    if layout == xs.XS_LAYOUT_A2A:
        outs = _shards(B, S, H, D, P)
    elif layout == xs.XS_LAYOUT_CONTIGUOUS:
        outs = [torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")]
    else:
        outs = [torch.full((B, S, H // P, D), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    xs.xs_attn_fwd_balanced(q, k, v, layout, outs, scale, ws)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    return outs


@pytest.mark.parametrize("S,D,P,B,H", SHAPES, ids=[f"S{c[0]}_D{c[1]}_P{c[2]}_B{c[3]}_H{c[4]}" for c in SHAPES])
def test_balanced_vs_oracle(xs, S, D, P, B, H):
    import oracle
    splits = _check_splits(B, S, H)
    if H == 5 and S == 4096:
        assert max(len(c) for c in splits.values()) >= 3, "some tile must be cut into four pieces"
    nbytes = xs.xs_attn_workspace_bytes(B, S, H, D)
    assert nbytes >= _sms() * (128 * D * 4 + 128 * 8 + 32)
    ws = xs.Workspace(nbytes)
    w = di.Workload("bal", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=S + D)
    qb, kb, vb = di.random_qkv(w)
    q, k, v = (bits_to_torch(x) for x in (qb, kb, vb))
    outs = _run(xs, q, k, v, w.scale, P, ws)
    got = np.stack([torch_to_f64(o) for o in outs])
    ref = oracle.attention_a2a(qb, kb, vb, w.scale, P)
    mass = oracle.attention_a2a(qb, kb, abs_bits(vb), w.scale, P)
    assert_close(got, ref, mass, f"balanced S={S} H={H}")
    # the plain schedule on the same inputs agrees to rounding
    plain = _shards(B, S, H, D, P)
    xs.xs_attn_a2a_fwd(q, k, v, plain, w.scale)
    torch.cuda.synchronize()
    diff = max(float((a.float() - b.float()).abs().max()) for a, b in zip(outs, plain))
    assert diff <= 2e-2


def test_balanced_layouts_bit_identical(xs):
    S, D, P, B, H = SHAPES[2]
    _check_splits(B, S, H)
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    w = di.Workload("lay", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=7)
    q, k, v = (bits_to_torch(x) for x in di.random_qkv(w))
    fused = _run(xs, q, k, v, w.scale, P, ws, xs.XS_LAYOUT_A2A)
    cont = _run(xs, q, k, v, w.scale, P, ws, xs.XS_LAYOUT_CONTIGUOUS)[0]
    heads = _run(xs, q, k, v, w.scale, P, ws, xs.XS_LAYOUT_HEADS)
    serial = _shards(B, S, H, D, P)
    xs.xs_relayout_a2a(heads, serial)
    torch.cuda.synchronize()
    Sl = S // P
    for p in range(P):
        assert torch.equal(fused[p].view(torch.int16), cont[:, p * Sl:(p + 1) * Sl].view(torch.int16))
        assert torch.equal(fused[p].view(torch.int16), serial[p].view(torch.int16))


def test_balanced_deterministic_and_workspace_reuse(xs):
    """Back-to-back launches on one workspace: flags left by the previous launch
    must not be taken for the current one's (each launch has its own epoch)."""
    import oracle
    S, D, P, B, H = SHAPES[1]
    _check_splits(B, S, H)
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    wa = di.Workload("a", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=11)
    wb = di.Workload("b", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=12)
    a = [bits_to_torch(x) for x in di.random_qkv(wa)]
    bb = di.random_qkv(wb)
    b = [bits_to_torch(x) for x in bb]
    r1 = _run(xs, *a, wa.scale, P, ws)
    r2 = _run(xs, *b, wb.scale, P, ws)
    r3 = _run(xs, *a, wa.scale, P, ws)
    for x, y in zip(r1, r3):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    ref = oracle.attention_a2a(*bb, wb.scale, P)
    mass = oracle.attention_a2a(bb[0], bb[1], abs_bits(bb[2]), wb.scale, P)
    assert_close(np.stack([torch_to_f64(o) for o in r2]), ref, mass, "second input on a reused workspace")


@pytest.mark.parametrize("S,D,P,H", [(4000, 128, 5, 5), (32768, 128, 4, 12)])
def test_balanced_layout_bit_exact(xs, S, D, P, H):
    B = 1
    _check_splits(B, S, H)     # 32768 x 12 heads: the small video-DiT shape
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
    outs = _run(xs, q, k, v, scale, P, ws)
    Sl = S // P
    for p in range(P):
        exp = di.layout_code_value_torch(B, S, H, D, s_offset=p * Sl, S_rows=Sl)
        eq = outs[p].view(torch.int16) == exp.view(torch.int16)
        assert bool(eq.all()), f"shard {p}: {int((~eq).sum())} elements differ"


def test_balanced_video_rows_of_split_tiles(xs):
    """Small video-DiT shape (3072 tiles, 32 left over after 20 whole waves):
    sampled rows plus three rows of every split tile."""
    import oracle
    w = di.WORKLOADS["video_small"]
    n = (w.S + 127) // 128
    splits = split_tiles(w.B * w.H * n, n, _sms())
    assert splits
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(w.B, w.S, w.H, w.D))
    qb, kb, vb = di.random_qkv(w)
    outs = _run(xs, *(bits_to_torch(x) for x in (qb, kb, vb)), w.scale, w.P, ws)
    rb, rs = di.sample_rows(w, 64)
    rows = set(zip(rb.tolist(), rs.tolist()))
    for t in splits:
        qt = t % n
        b = t // (n * w.H)
        for r in (0, 61, 127):
            rows.add((b, min(qt * 128 + r, w.S - 1)))
    rows = sorted(rows)
    rb = np.array([r[0] for r in rows], dtype=np.int64)
    rs = np.array([r[1] for r in rows], dtype=np.int64)
    ref = oracle.attention_rows(qb, kb, vb, w.scale, rb, rs)
    mass = oracle.attention_rows(qb, kb, abs_bits(vb), w.scale, rb, rs)
    Sl = w.S // w.P
    got = np.stack([torch_to_f64(outs[int(s) // Sl][int(b), int(s) % Sl]) for b, s in zip(rb, rs)])
    assert_close(got, ref, mass, "video_small balanced")


def test_workspace_too_small_is_refused(xs):
    S, D, P, B, H = SHAPES[0]
    need = xs.xs_attn_workspace_bytes(B, S, H, D)
    small = xs.Workspace(need - 256)
    q = torch.zeros((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    outs = _shards(B, S, H, D, P)
    with pytest.raises(xs.XsError) as e:
        xs.xs_attn_fwd_balanced(q, q, q, xs.XS_LAYOUT_A2A, outs, 0.1, small)
    assert e.value.code == xs.XS_ERR_WORKSPACE


def test_no_workspace_needed_when_waves_are_whole(xs):
    G = _sms()
    S, D, B = 128 * G, 128, 1          # H = 1: exactly G tiles
    assert xs.xs_attn_workspace_bytes(B, S, 1, D) == 0
    assert xs.xs_attn_workspace_bytes(1, 256, 2, 64) == 0   # 4 tiles of 2 blocks: nothing to gain
    assert xs.xs_attn_workspace_bytes(1, 1024, 20, 128) == 0  # 8 left over tiles of 8 blocks
    assert xs.xs_attn_workspace_bytes(1, 4608, 24, 128) == 0  # image-DiT: too little to gain


def test_balanced_expired_wait_is_reported(xs, monkeypatch):
    import oracle
    S, D, P, B, H = SHAPES[0]
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    w = di.Workload("wl", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=3)
    qb, kb, vb = di.random_qkv(w)
    q, k, v = (bits_to_torch(x) for x in (qb, kb, vb))
    outs = _shards(B, S, H, D, P, fill=0.0)
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    monkeypatch.setenv("XSATTN_WAIT_TIMEOUT_NS", "0")
    xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, outs, w.scale, ws)
    assert xs.xs_attn_get_device_error() == xs.XS_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("XSATTN_WAIT_TIMEOUT_NS")
    outs = _run(xs, q, k, v, w.scale, P, ws)
    ref = oracle.attention_a2a(qb, kb, vb, w.scale, P)
    mass = oracle.attention_a2a(qb, kb, abs_bits(vb), w.scale, P)
    assert_close(np.stack([torch_to_f64(o) for o in outs]), ref, mass, "balanced after timeout")


def test_staged_host_entry_with_workspace_vs_oracle(xs):
    """xs_attn_a2a_fwd_staged with a workspace: the head groups of its pipeline
    run the balanced schedule planned for their own heads (here every one-head
    group splits its 32 tiles over 128 CTAs), so its split tiles are merged in a
    different order than the whole-shape call's: checked against the oracle and
    against the device-side call to rounding."""
    import oracle
    S, D, P, B, H = SHAPES[0]
    _check_splits(B, S, H)
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    w = di.Workload("st", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=17)
    bits = di.random_qkv(w)
    qd, kd, vd = (bits_to_torch(x) for x in bits)
    ref = _run(xs, qd, kd, vd, w.scale, P, ws)
    pin = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = (pin(x) for x in bits)
    out_h = [torch.empty((B, S // P, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(P)]
    out_d = _shards(B, S, H, D, P)
    xs.xs_attn_a2a_fwd_staged(qh, kh, vh, out_h, qd, kd, vd, out_d, w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert xs.xs_attn_get_device_error() == xs.XS_OK
    got = np.stack([torch_to_f64(o) for o in out_h])
    exp = oracle.attention_a2a(*bits, w.scale, P)
    mass = oracle.attention_a2a(bits[0], bits[1], abs_bits(bits[2]), w.scale, P)
    assert_close(got, exp, mass, "staged with a workspace")
    assert max(float((a.float() - b.cpu().float()).abs().max()) for a, b in zip(out_h, ref)) <= 2e-2


def test_balanced_graph_replay_takes_only_its_own_flags(xs):
    """One split launch captured in a CUDA graph and replayed three times with
    different inputs copied into the captured buffers: every replay must merge
    the partial results of its own launch only.  The flags' epoch comes from the
    workspace's launch count, not from the captured arguments, so each replay
    matches an uncaptured call on the same inputs bit for bit."""
    S, D, P, B, H = SHAPES[0]
    _check_splits(B, S, H)
    ws = xs.Workspace(xs.xs_attn_workspace_bytes(B, S, H, D))
    wa = di.Workload("ga", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=31)
    wb = di.Workload("gb", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=32)
    a = [bits_to_torch(x) for x in di.random_qkv(wa)]
    b = [bits_to_torch(x) for x in di.random_qkv(wb)]
    ref_a = _run(xs, *a, wa.scale, P, ws)
    ref_b = _run(xs, *b, wa.scale, P, ws)
    q, k, v = (torch.empty_like(x) for x in a)
    outs = _shards(B, S, H, D, P)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        xs.xs_attn_fwd_balanced(q, k, v, xs.XS_LAYOUT_A2A, outs, wa.scale, ws)
    for src, ref in ((a, ref_a), (b, ref_b), (a, ref_a)):
        for dst, x in zip((q, k, v), src):
            dst.copy_(x)
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert xs.xs_attn_get_device_error() == xs.XS_OK
        for x, y in zip(outs, ref):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
