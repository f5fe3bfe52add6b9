"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each test fixes the oracle to something the mathematics or a hand derivation
determines: a hand-worked example, closed forms (Q = 0, scale = 0, one-hot
rows), invariants (row sums, key permutation, key shift, query permutation),
brute force with an independent full-matrix NumPy evaluation and 50-digit
mpmath, a library cross-check (torch CPU fp64 SDPA) and a hand-written index
table of the Ulysses All-to-All.  None of these needs a GPU.
"""
import math
import os

import numpy as np
import pytest

import dit_inputs as di
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return di.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _f64(bits):
    return di.bf16_bits_to_f32(bits).astype(np.float64)


def _rand(shape, seed, grid=None):
    x = np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
    if grid:
        x = np.clip(np.round(x * grid) / grid, -4, 4).astype(np.float32)
    return _bits(x)


def _brute_numpy(q, k, v, scale):
    """Full S x S evaluation with NumPy: materialise every score matrix."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    x = np.einsum("bihd,bjhd->bhij", qf, kf) * scale
    w = np.exp(x - x.max(axis=-1, keepdims=True))
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("bhij,bjhd->bihd", w, vf)


# ------------------------------------------------------------------ golden
def test_worked_example_by_hand():
    recs = [ln.split() for ln in open(os.path.join(GOLDEN, "worked_example_attention.txt"))
            if ln.strip() and not ln.startswith("#")]
    scale = float(next(r[1] for r in recs if r[0] == "scale"))
    t = {n: np.zeros((1, 3, 1, 2), dtype=np.float64) for n in "qkvo"}
    for r in recs:
        if r[0] in t:
            t[r[0]][0, int(r[1]), 0, int(r[2])] = float(r[3])
    o = oracle.attention(_bits(t["q"]), _bits(t["k"]), _bits(t["v"]), scale)
    np.testing.assert_allclose(o, t["o"], rtol=0, atol=1e-14)


def test_reshard_index_table_by_hand():
    B, S, H, D, P = 2, 4, 2, 1, 2
    O = np.zeros((B, S, H, D))
    for b in range(B):
        for s in range(S):
            for h in range(H):
                O[b, s, h, 0] = 100 * b + 10 * s + h
    L = oracle.head_shards(O, P)
    for r in range(P):
        np.testing.assert_array_equal(L[r][..., 0, 0], O[:, :, r, 0])
    out = oracle.a2a(L)
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "ulysses_reshard_index_table.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == P * B * (S // P) * H
    for p, b, s2, h, val in (map(int, r) for r in rows):
        assert out[p, b, s2, h, 0] == val, (p, b, s2, h)


def test_head_shards_hold_contiguous_head_ranges():
    """H = 4, P = 2: rank 0 holds heads 0 and 1, rank 1 holds heads 2 and 3, in
    that order; every destination shard holds all four heads in global order."""
    B, S, H, D, P = 1, 2, 4, 1, 2
    O = np.zeros((B, S, H, D))
    O[0, :, :, 0] = [[0, 1, 2, 3], [10, 11, 12, 13]]   # O[b,s,h] = 10*s + h
    L = oracle.head_shards(O, P)
    np.testing.assert_array_equal(L[0, 0, :, :, 0], [[0, 1], [10, 11]])
    np.testing.assert_array_equal(L[1, 0, :, :, 0], [[2, 3], [12, 13]])
    out = oracle.a2a(L)
    np.testing.assert_array_equal(out[0, 0, :, :, 0], [[0, 1, 2, 3]])
    np.testing.assert_array_equal(out[1, 0, :, :, 0], [[10, 11, 12, 13]])


# ------------------------------------------------------------- brute force
@pytest.mark.parametrize("S", [1, 2, 3, 8, 64, 200])
@pytest.mark.parametrize("H", [1, 2, 4])
def test_brute_force_numpy(S, H):
    B, D = 2, 16
    q, k, v = (_rand((B, S, H, D), 10 * S + H + i) for i in range(3))
    scale = 1 / math.sqrt(D)
    ref = _brute_numpy(q, k, v, scale)
    got = oracle.attention(q, k, v, scale, nthreads=2)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("S", [1, 2, 3, 5, 8])
def test_brute_force_mpmath_50_digits(S):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    B, H, D = 1, 2, 4
    q, k, v = (_rand((B, S, H, D), 77 + S + i) for i in range(3))
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    scale = 0.37
    got = oracle.attention(q, k, v, scale)
    for h in range(H):
        for i in range(S):
            x = [mp.mpf(scale) * mp.fsum(mp.mpf(qf[0, i, h, d]) * mp.mpf(kf[0, j, h, d]) for d in range(D))
                 for j in range(S)]
            m = max(x)
            w = [mp.exp(xj - m) for xj in x]
            l = mp.fsum(w)
            for d in range(D):
                ref = mp.fsum(w[j] * mp.mpf(vf[0, j, h, d]) for j in range(S)) / l
                assert abs(got[0, i, h, d] - float(ref)) <= 1e-13 * max(1.0, abs(float(ref)))


# ------------------------------------------------------------ closed forms
@pytest.mark.parametrize("S", [1, 7, 130])
def test_q_zero_gives_mean_of_v(S):
    B, H, D = 2, 3, 8
    q = np.zeros((B, S, H, D), dtype=np.uint16)  # +0.0 in bf16
    k, v = _rand((B, S, H, D), 5), _rand((B, S, H, D), 6)
    got = oracle.attention(q, k, v, 0.125)
    mean = _f64(v).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(got, np.broadcast_to(mean, got.shape), rtol=1e-12, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    B, S, H, D = 1, 33, 2, 8
    q, k, v = (_rand((B, S, H, D), 40 + i) for i in range(3))
    got = oracle.attention(q, k, v, 0.0)
    mean = _f64(v).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(got, np.broadcast_to(mean, got.shape), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("B,S,H,D", [(1, 256, 2, 64), (2, 96, 4, 64), (1, 1000, 2, 128), (1, 1024, 1, 64)])
def test_one_hot_rows_copy_own_value_row(B, S, H, D):
    """Index-coded Q = K with a large scale: every row's softmax is one-hot on
    its own key, so O = V exactly (the expected value is the encoding itself).
    S = 1024 at D = 64 takes the code with 4 channels per bit."""
    q, k, v, scale = di.layout_code_inputs(B, S, H, D)
    got = oracle.attention(q, k, v, scale)
    # every other key trails the own key by >= 2 * (channels per bit) in q.k, so
    # its weight is <= exp(-gap*scale); with values < 256 the exact output differs
    # from the own value row by less than S * 256 * exp(-gap*scale)
    gap = 14 if math.ceil(math.log2(S)) * 7 <= D else 8
    bound = S * 256 * math.exp(-gap * scale)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(got[b, :, h, :],
                                       di.layout_code_value(b, np.arange(S), h, D).astype(np.float64),
                                       rtol=0, atol=bound)


# -------------------------------------------------------------- invariants
def test_weights_sum_to_one_and_match_output():
    B, S, H, D = 2, 300, 3, 32
    q, k, v = (_rand((B, S, H, D), 90 + i) for i in range(3))
    full = oracle.attention(q, k, v, 0.3)
    for (b, i, h) in [(0, 0, 0), (1, 299, 2), (1, 17, 1)]:
        w, orow = oracle.attention_weights(q, k, v, 0.3, b, i, h)
        assert np.all(w >= 0)
        assert abs(w.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(orow, full[b, i, h], rtol=1e-13, atol=1e-15)
        # the output row is a convex combination of value rows
        vf = _f64(v)[b, :, h, :]
        assert np.all(orow <= vf.max(axis=0) + 1e-12) and np.all(orow >= vf.min(axis=0) - 1e-12)


def test_key_permutation_invariance():
    B, S, H, D = 1, 150, 2, 16
    q, k, v = (_rand((B, S, H, D), 20 + i) for i in range(3))
    perm = np.random.default_rng(3).permutation(S)
    a = oracle.attention(q, k, v, 0.25)
    b = oracle.attention(q, k[:, perm], v[:, perm], 0.25)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    # permuting only V (not K) must change the result: K and V rows are paired
    c = oracle.attention(q, k, v[:, perm], 0.25)
    assert np.abs(a - c).max() > 1e-3


def test_query_permutation_equivariance():
    B, S, H, D = 1, 120, 2, 16
    q, k, v = (_rand((B, S, H, D), 30 + i) for i in range(3))
    perm = np.random.default_rng(4).permutation(S)
    a = oracle.attention(q, k, v, 0.25)
    b = oracle.attention(q[:, perm], k, v, 0.25)
    np.testing.assert_allclose(a[:, perm], b, rtol=1e-12, atol=1e-14)


def test_key_shift_invariance():
    """Adding the same vector u to every key shifts each row's scores by a
    constant (scale * q.u), which softmax ignores."""
    B, S, H, D = 1, 90, 2, 16
    q = _rand((B, S, H, D), 50, grid=8)
    k = _rand((B, S, H, D), 51, grid=8)
    v = _rand((B, S, H, D), 52)
    u = np.zeros(D, dtype=np.float32)
    u[::3] = 1.0
    k_shift = _bits(di.bf16_bits_to_f32(k) + u)  # exact: grid 1/8 values within [-4, 5]
    np.testing.assert_array_equal(di.bf16_bits_to_f32(k_shift) - di.bf16_bits_to_f32(k),
                                  np.broadcast_to(u, k.shape))
    a = oracle.attention(q, k, v, 0.3)
    b = oracle.attention(q, k_shift, v, 0.3)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-13)


def test_heads_and_batches_are_independent():
    B, S, H, D = 2, 64, 3, 8
    q, k, v = (_rand((B, S, H, D), 60 + i) for i in range(3))
    full = oracle.attention(q, k, v, 0.5)
    for b in range(B):
        for h in range(H):
            one = oracle.attention(q[b:b + 1, :, h:h + 1].copy(), k[b:b + 1, :, h:h + 1].copy(),
                                   v[b:b + 1, :, h:h + 1].copy(), 0.5)
            np.testing.assert_array_equal(one[0, :, 0], full[b, :, h])


# ------------------------------------------------------- library cross-check
def test_torch_sdpa_fp64_crosscheck():
    torch = pytest.importorskip("torch")
    B, S, H, D = 2, 257, 4, 64
    q, k, v = (_rand((B, S, H, D), 70 + i) for i in range(3))
    scale = 1 / math.sqrt(D)
    t = [torch.from_numpy(_f64(x)).permute(0, 2, 1, 3) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=scale).permute(0, 2, 1, 3).numpy()
    got = oracle.attention(q, k, v, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------- re-shard
@pytest.mark.parametrize("B,S,H,P", [(1, 8, 4, 2), (2, 12, 6, 3), (1, 16, 8, 8), (2, 6, 2, 1)])
def test_a2a_round_trip_and_permutation(B, S, H, P):
    D = 3
    L = np.random.default_rng(B * 100 + S).standard_normal((P, B, S, H // P, D))
    out = oracle.a2a(L)
    assert out.shape == (P, B, S // P, H, D)
    np.testing.assert_array_equal(oracle.a2a_inverse(out), L)
    np.testing.assert_array_equal(np.sort(out, axis=None), np.sort(L, axis=None))


def test_reshard_of_one_hot_layout_inputs():
    """End-to-end oracle path on the index-coded inputs: shard p, row s' must
    hold the encoding of the global row p*S/P + s' for every head."""
    B, S, H, D, P = 2, 256, 8, 64, 4
    q, k, v, scale = di.layout_code_inputs(B, S, H, D)
    out = oracle.attention_a2a(q, k, v, scale, P)
    bound = S * 256 * math.exp(-14 * scale)
    Sl = S // P
    for p in range(P):
        for b in range(B):
            for h in range(H):
                exp = di.layout_code_value(b, p * Sl + np.arange(Sl), h, D)
                np.testing.assert_allclose(out[p, b, :, h, :], exp.astype(np.float64), rtol=0, atol=bound)


def test_rows_entry_matches_full():
    w = di.Workload("t", B=2, H=3, S=200, D=32, P=4, scale=0.2)
    q, k, v = di.random_qkv(w)
    full = oracle.attention(q, k, v, w.scale)
    rb, rs = di.sample_rows(w, 40)
    rows = oracle.attention_rows(q, k, v, w.scale, rb, rs)
    np.testing.assert_array_equal(rows, full[rb, rs])


def test_argument_errors():
    o = np.zeros((1, 4, 3, 2))
    with pytest.raises(ValueError):
        oracle.head_shards(o, 2)          # H % P != 0
    with pytest.raises(TypeError):
        oracle.attention(np.zeros((1, 2, 1, 2), np.float32), *[np.zeros((1, 2, 1, 2), np.uint16)] * 2, 1.0)


# ------------------------------------------------------------ Ulysses step
@pytest.mark.parametrize("B,S,H,D,P", [(2, 16, 4, 8, 2), (1, 24, 8, 4, 4), (1, 9, 3, 8, 3)])
def test_ulysses_step_equals_attention_on_the_whole_sequence(B, S, H, D, P):
    """The three-step Ulysses oracle (pre-attention exchange, per-rank attention on
    its heads, post-attention exchange) against brute force on the whole sequence,
    re-sharded by plain slicing: sequence shard p holds rows [p*S/P, (p+1)*S/P)
    of every head."""
    q, k, v = (_rand((B, S, H, D), seed) for seed in (31, 32, 33))
    Sl = S // P
    shards = [np.stack([x[:, p * Sl:(p + 1) * Sl] for p in range(P)]) for x in (q, k, v)]
    got = oracle.ulysses_attention(*shards, 0.7)
    full = _brute_numpy(q, k, v, 0.7)
    want = np.stack([full[:, p * Sl:(p + 1) * Sl] for p in range(P)])
    assert got.shape == (P, B, Sl, H, D)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_ulysses_step_shard_order_equivariance_and_key_value_pairing():
    """Renumbering the ranks (the same shard order for Q, K and V) renumbers the
    output shards; giving K alone a different order breaks the key/value pairing
    and must change the result."""
    B, S, H, D, P = 1, 16, 4, 8, 4
    q, k, v = (_rand((B, S, H, D), seed) for seed in (41, 42, 43))
    Sl = S // P
    shards = [np.stack([x[:, p * Sl:(p + 1) * Sl] for p in range(P)]) for x in (q, k, v)]
    good = oracle.ulysses_attention(*shards, 0.5)
    rev = oracle.ulysses_attention(*[x[::-1].copy() for x in shards], 0.5)
    np.testing.assert_allclose(rev[::-1], good, rtol=1e-12, atol=1e-12)
    k_only = oracle.ulysses_attention(shards[0], shards[1][::-1].copy(), shards[2], 0.5)
    assert np.abs(k_only - good).max() > 1e-3
