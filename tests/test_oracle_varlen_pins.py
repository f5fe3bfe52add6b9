"""Pins for the oracle's packed variable-length attention (attention_varlen):
sequences of given lengths lie back to back in one [1, T, H, D] tensor and each
query row attends only to its own sequence (causal: up to its own position).
Not on the X-Stage pages; the usual variable-length batch of attention kernels.

Pinned to a hand-worked example, a masked full-matrix NumPy evaluation, a
library cross-check (torch fp64 SDPA with a block-diagonal mask), and
structural facts: one sequence is plain attention, equal lengths are batched
attention, other sequences and empty sequences do not matter, and Q = 0 gives
per-sequence (prefix) means of V.  A segment boundary off by one row, or rows
attending across sequences, fails several of them.
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


def _seq_ids(seqlens):
    return np.repeat(np.arange(len(seqlens)), seqlens)


def _mask(seqlens, causal):
    sid = _seq_ids(seqlens)
    m = sid[:, None] == sid[None, :]
    if causal:
        m &= np.tri(len(sid), len(sid), dtype=bool)
    return m


def _brute_numpy(q, k, v, seqlens, scale, causal):
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    x = np.einsum("bihd,bjhd->bhij", qf, kf) * scale
    x = np.where(_mask(seqlens, causal), x, -np.inf)
    w = np.exp(x - x.max(axis=-1, keepdims=True))
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("bhij,bjhd->bihd", w, vf)


MIXES = [[1, 2], [5, 1, 7], [64, 3, 0, 30], [130, 1, 127, 129], [200]]


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_worked_example_by_hand(causal):
    recs = [ln.split() for ln in open(os.path.join(GOLDEN, "worked_example_varlen_attention.txt"))
            if ln.strip() and not ln.startswith("#")]
    seqlens = [int(x) for x in next(r[1:] for r in recs if r[0] == "seqlens")]
    scale = float(next(r[1] for r in recs if r[0] == "scale"))
    t = {n: np.zeros((1, 3, 1, 2), dtype=np.float64) for n in ("q", "k", "v", "o", "oc")}
    for r in recs:
        if r[0] in t:
            t[r[0]][0, int(r[1]), 0, int(r[2])] = float(r[3])
    got = oracle.attention_varlen(_bits(t["q"]), _bits(t["k"]), _bits(t["v"]), seqlens, scale, causal=causal)
    np.testing.assert_allclose(got, t["oc" if causal else "o"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seqlens", MIXES, ids=["-".join(map(str, m)) for m in MIXES])
def test_varlen_brute_force_numpy(seqlens, causal):
    T, H, D = sum(seqlens), 2, 16
    q, k, v = (_rand((1, T, H, D), 10 * T + i) for i in range(3))
    got = oracle.attention_varlen(q, k, v, seqlens, 0.25, causal=causal)
    np.testing.assert_allclose(got, _brute_numpy(q, k, v, seqlens, 0.25, causal), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_torch_sdpa_fp64_crosscheck(causal):
    torch = pytest.importorskip("torch")
    seqlens = [100, 1, 57, 99]
    T, H, D = sum(seqlens), 3, 64
    q, k, v = (_rand((1, T, H, D), 200 + i) for i in range(3))
    t = [torch.from_numpy(_f64(x)).permute(0, 2, 1, 3) for x in (q, k, v)]
    mask = torch.from_numpy(_mask(seqlens, causal))
    ref = torch.nn.functional.scaled_dot_product_attention(*t, attn_mask=mask, scale=1 / math.sqrt(D))
    got = oracle.attention_varlen(q, k, v, seqlens, 1 / math.sqrt(D), causal=causal)
    np.testing.assert_allclose(got, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_one_sequence_is_plain_attention(causal):
    q, k, v = (_rand((1, 150, 2, 16), 300 + i) for i in range(3))
    np.testing.assert_array_equal(oracle.attention_varlen(q, k, v, [150], 0.3, causal=causal),
                                  oracle.attention(q, k, v, 0.3, causal=causal))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equal_lengths_are_batched_attention(causal):
    B, S, H, D = 3, 40, 2, 16
    q, k, v = (_rand((B, S, H, D), 310 + i) for i in range(3))
    packed = [x.reshape(1, B * S, H, D) for x in (q, k, v)]
    got = oracle.attention_varlen(*packed, [S] * B, 0.3, causal=causal)
    np.testing.assert_array_equal(got.reshape(B, S, H, D), oracle.attention(q, k, v, 0.3, causal=causal))


def test_varlen_other_and_empty_sequences_do_not_matter():
    seqlens = [30, 45, 20]
    T, H, D = sum(seqlens), 2, 16
    q, k, v = (_rand((1, T, H, D), 320 + i) for i in range(3))
    a = oracle.attention_varlen(q, k, v, seqlens, 0.4)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x, seed in ((q2, 1), (k2, 2), (v2, 3)):   # new contents for sequences 0 and 2
        x[:, :30] = _rand((1, 30, H, D), 400 + seed)
        x[:, 75:] = _rand((1, 20, H, D), 410 + seed)
    b = oracle.attention_varlen(q2, k2, v2, seqlens, 0.4)
    np.testing.assert_array_equal(a[:, 30:75], b[:, 30:75])
    assert not np.allclose(a[:, :30], b[:, :30]) and not np.allclose(a[:, 75:], b[:, 75:])
    np.testing.assert_array_equal(oracle.attention_varlen(q, k, v, [0, 30, 0, 0, 45, 20, 0], 0.4), a)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_q_zero_gives_sequence_means(causal):
    seqlens = [1, 9, 20]
    T, H, D = sum(seqlens), 2, 8
    q = np.zeros((1, T, H, D), dtype=np.uint16)
    k, v = _rand((1, T, H, D), 330), _rand((1, T, H, D), 331)
    got = oracle.attention_varlen(q, k, v, seqlens, 0.5, causal=causal)
    vf = _f64(v)
    start = 0
    for n in seqlens:
        seg = vf[:, start:start + n]
        want = (np.cumsum(seg, axis=1) / np.arange(1, n + 1)[None, :, None, None] if causal
                else np.broadcast_to(seg.mean(axis=1, keepdims=True), seg.shape))
        np.testing.assert_allclose(got[:, start:start + n], want, rtol=1e-12, atol=1e-14)
        start += n


def test_varlen_argument_errors():
    x = np.zeros((1, 5, 1, 2), np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_varlen(x, x, x, [2, 2], 1.0)       # lengths do not sum to T
    with pytest.raises(ValueError):
        oracle.attention_varlen(x, x, x, [6, -1], 1.0)      # negative length
    with pytest.raises(ValueError):
        oracle.attention_varlen(np.zeros((2, 5, 1, 2), np.uint16), x, x, [5], 1.0)
