"""Pins for the causal variant of the CPU oracle (row i attends to keys 0 .. i).

The causal form is not on the X-Stage pages (they treat bidirectional DiT
attention); it is the masked self-attention of autoregressive models.  Each
test fixes the oracle's causal entries to something other than the oracle: a
hand-worked example, closed forms (the first row copies the first value row;
Q = 0 gives prefix means of V), invariants (future keys and values do not
matter, the last row equals bidirectional attention, weights vanish above the
diagonal and sum to 1), brute force with a masked full-matrix NumPy evaluation
and a library cross-check (torch CPU fp64 SDPA with is_causal).  A mask that
is off by one key, reversed or ignored fails several of them.
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


def _rand(shape, seed):
    return _bits(np.random.default_rng(seed).standard_normal(shape).astype(np.float32))


def _brute_numpy_causal(q, k, v, scale):
    """Full S x S scores with NumPy, keys above the diagonal set to -inf."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    S = qf.shape[1]
    x = np.einsum("bihd,bjhd->bhij", qf, kf) * scale
    x = np.where(np.tri(S, S, dtype=bool), x, -np.inf)
    w = np.exp(x - x.max(axis=-1, keepdims=True))
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("bhij,bjhd->bihd", w, vf)


def test_causal_worked_example_by_hand():
    recs = [ln.split() for ln in open(os.path.join(GOLDEN, "worked_example_causal_attention.txt"))
            if ln.strip() and not ln.startswith("#")]
    scale = float(next(r[1] for r in recs if r[0] == "scale"))
    t = {n: np.zeros((1, 3, 1, 2), dtype=np.float64) for n in "qkvo"}
    for r in recs:
        if r[0] in t:
            t[r[0]][0, int(r[1]), 0, int(r[2])] = float(r[3])
    o = oracle.attention(_bits(t["q"]), _bits(t["k"]), _bits(t["v"]), scale, causal=True)
    np.testing.assert_allclose(o, t["o"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("S", [1, 5, 130])
def test_causal_first_row_copies_first_value_row(S):
    B, H, D = 2, 3, 16
    q, k, v = (_rand((B, S, H, D), 40 + i) for i in range(3))
    got = oracle.attention(q, k, v, 0.3, causal=True)
    np.testing.assert_array_equal(got[:, 0], _f64(v)[:, 0])   # one key: weight exactly 1


@pytest.mark.parametrize("S", [1, 7, 130])
def test_causal_q_zero_gives_prefix_means_of_v(S):
    B, H, D = 2, 3, 8
    q = np.zeros((B, S, H, D), dtype=np.uint16)
    k, v = _rand((B, S, H, D), 5), _rand((B, S, H, D), 6)
    got = oracle.attention(q, k, v, 0.125, causal=True)
    vf = _f64(v)
    prefix_mean = np.cumsum(vf, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(got, prefix_mean, rtol=1e-12, atol=1e-14)


def test_causal_last_row_equals_bidirectional():
    B, S, H, D = 2, 67, 3, 32
    q, k, v = (_rand((B, S, H, D), 50 + i) for i in range(3))
    causal = oracle.attention(q, k, v, 0.2, causal=True)
    full = oracle.attention(q, k, v, 0.2)
    np.testing.assert_array_equal(causal[:, -1], full[:, -1])
    assert not np.allclose(causal[:, 0], full[:, 0])


def test_causal_future_keys_and_values_do_not_matter():
    B, S, H, D, i = 1, 40, 2, 16, 23
    q, k, v = (_rand((B, S, H, D), 60 + n) for n in range(3))
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1:] = _rand((B, S - i - 1, H, D), 70)
    v2[:, i + 1:] = _rand((B, S - i - 1, H, D), 71)
    a = oracle.attention(q, k, v, 0.25, causal=True)
    b = oracle.attention(q, k2, v2, 0.25, causal=True)
    np.testing.assert_array_equal(a[:, :i + 1], b[:, :i + 1])
    assert not np.allclose(a[:, i + 1:], b[:, i + 1:])
    # a change at key i itself must reach row i
    k3 = k.copy()
    k3[:, i] = _rand((B, 1, H, D), 72)[:, 0]
    c = oracle.attention(q, k3, v, 0.25, causal=True)
    np.testing.assert_array_equal(a[:, :i], c[:, :i])
    assert not np.allclose(a[:, i], c[:, i])


def test_causal_weights_vanish_above_the_diagonal_and_sum_to_one():
    B, S, H, D = 1, 33, 2, 16
    q, k, v = (_rand((B, S, H, D), 80 + n) for n in range(3))
    full = oracle.attention(q, k, v, 0.5, causal=True)
    for i in (0, 1, 16, 32):
        w, o = oracle.attention_weights(q, k, v, 0.5, 0, i, 1, causal=True)
        assert np.all(w[i + 1:] == 0.0) and np.all(w[:i + 1] > 0.0)
        assert abs(w.sum() - 1.0) < 1e-12
        np.testing.assert_allclose(w @ _f64(v)[0, :, 1], o, rtol=1e-12, atol=1e-14)
        np.testing.assert_array_equal(o, full[0, i, 1])


@pytest.mark.parametrize("S", [1, 2, 3, 8, 64, 200])
def test_causal_brute_force_numpy(S):
    B, H, D = 2, 2, 16
    q, k, v = (_rand((B, S, H, D), 90 + S + i) for i in range(3))
    scale = 1 / math.sqrt(D)
    np.testing.assert_allclose(oracle.attention(q, k, v, scale, nthreads=2, causal=True),
                               _brute_numpy_causal(q, k, v, scale), rtol=1e-12, atol=1e-13)


def test_causal_torch_sdpa_fp64_crosscheck():
    torch = pytest.importorskip("torch")
    B, S, H, D = 2, 257, 4, 64
    q, k, v = (_rand((B, S, H, D), 100 + i) for i in range(3))
    scale = 1 / math.sqrt(D)
    t = [torch.from_numpy(_f64(x)).permute(0, 2, 1, 3) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=scale, is_causal=True)
    got = oracle.attention(q, k, v, scale, causal=True)
    np.testing.assert_allclose(got, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-11, atol=1e-13)


def test_causal_rows_entry_matches_full():
    w = di.Workload("t", B=2, H=3, S=200, D=32, P=4, scale=0.2)
    q, k, v = di.random_qkv(w)
    full = oracle.attention(q, k, v, w.scale, causal=True)
    rb, rs = di.sample_rows(w, 40)
    np.testing.assert_array_equal(oracle.attention_rows(q, k, v, w.scale, rb, rs, causal=True), full[rb, rs])


def test_causal_reshard_of_layout_code_inputs():
    """Index-coded inputs: every query's own key dominates and lies inside the
    causal window, so shard p, row s' still holds the encoding of global row
    p*S/P + s' (row 0 sees only itself and is exact)."""
    B, S, H, D, P = 2, 256, 8, 64, 4
    q, k, v, scale = di.layout_code_inputs(B, S, H, D)
    out = oracle.attention_a2a(q, k, v, scale, P, causal=True)
    bound = S * 256 * math.exp(-14 * scale)
    Sl = S // P
    for p in range(P):
        for b in range(B):
            for h in range(H):
                exp = di.layout_code_value(b, p * Sl + np.arange(Sl), h, D)
                np.testing.assert_allclose(out[p, b, :, h, :], exp.astype(np.float64), rtol=0, atol=bound)
