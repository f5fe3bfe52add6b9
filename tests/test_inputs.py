"""The seeded input generators: reproducible, correctly rounded, right shapes."""
import math

import numpy as np
import pytest

import dit_inputs as di


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37.0
    x[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8, 0.0]   # ties
    ours = di.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(di.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_random_qkv_reproducible_and_distinct():
    w = di.WORKLOADS["tiny"]
    a = di.random_qkv(w)
    b = di.random_qkv(w)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
        assert x.shape == (1, 256, 2, 64) and x.dtype == np.uint16
    assert not np.array_equal(a[0], a[1]) and not np.array_equal(a[1], a[2])
    f = di.bf16_bits_to_f32(a[0])
    assert abs(f.mean()) < 0.05 and abs(f.std() - 1) < 0.05


def test_outlier_channels_scaled():
    w = di.Workload("o", B=1, H=3, S=4096, D=128, P=1, scale=0.1, outliers=4)
    ch = di.outlier_channels(w)
    assert ch.shape == (3, 4)
    q, k, v = di.random_qkv(w)
    for t in (q, k, v):
        f = di.bf16_bits_to_f32(t)
        for h in range(3):
            std = f[0, :, h, :].std(axis=0)
            mask = np.zeros(128, bool)
            mask[ch[h]] = True
            assert np.all(std[mask] > 6) and np.all(std[~mask] < 1.2)


@pytest.mark.parametrize("S,D", [(256, 64), (1000, 128), (75776, 128), (1024, 64), (32768, 64)])
def test_layout_code_dot_products(S, D):
    q, k, v, scale = di.layout_code_inputs(1, S, 1, D)
    qf = di.bf16_bits_to_f32(q)[0, :, 0, :].astype(np.float64)
    rng = np.random.default_rng(S)
    s = rng.integers(0, S, 64)
    t = rng.integers(0, S, 64)
    dots = (qf[s] * qf[t]).sum(axis=1)
    ham = np.array([bin(int(a) ^ int(b)).count("1") for a, b in zip(s, t)])
    r = 7 if math.ceil(math.log2(S)) * 7 <= D else 4   # channels per bit
    np.testing.assert_array_equal(dots, D - 2 * r * ham)
    vf = di.bf16_bits_to_f32(v)[0, :, 0, :]
    np.testing.assert_array_equal(vf[s], di.layout_code_value(0, s, 0, D))


def test_sample_rows_cover_shard_edges():
    w = di.WORKLOADS["image"]
    b, s = di.sample_rows(w, 64)
    assert len(s) >= 64 and np.all(np.diff(b * w.S + s) > 0)
    for p in range(w.P):
        assert p * (w.S // w.P) in set(s) and (p + 1) * (w.S // w.P) - 1 in set(s)


def test_workload_table():
    assert di.WORKLOADS["video_large"].flops == 4 * 40 * 75776 ** 2 * 128
    assert di.SWEEP_S[0] == 1024 and di.SWEEP_S[-1] == 131072 and len(di.SWEEP_S) == 8


def test_layout_code_torch_matches_numpy():
    torch = pytest.importorskip("torch")
    for (B, S, H, D) in [(2, 256, 3, 64), (1, 1000, 2, 128)]:
        q, k, v, sc = di.layout_code_inputs(B, S, H, D)
        tq, tk, tv, tsc = di.layout_code_inputs_torch(B, S, H, D, device="cpu")
        assert sc == tsc
        for a, t in ((q, tq), (k, tk), (v, tv)):
            np.testing.assert_array_equal(a, t.view(torch.int16).numpy().view(np.uint16))
