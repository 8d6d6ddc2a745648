"""The seeded input generator: deterministic, correct shapes and recipe."""
import numpy as np
import pytest

from linear_cross_entropy_logit_gb300 import inputs as I


def test_bf16_rounding_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 1e-40, 3.0e38],
                    dtype=np.float32)
    bits = I.f32_to_bf16_bits(vals)
    back = I.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert back[0] == 1.0 and back[1] == 1.0
    # 1 + 3*2^-9 lies nearer 1 + 2^-7
    assert back[2] == np.float32(1.0 + 2 ** -7)
    assert back[3] == -2.5
    rel = np.abs(back - vals) / np.maximum(np.abs(vals), 1e-30)
    assert np.all(rel[4:] <= 2 ** -8)


def test_deterministic_and_seeded():
    spec = I.custom_spec("t", N=300, H=40, V=500, dtype="bf16", labels="zipf",
                         n_ignore=30, n_scaled_w_rows=5, w_row_scale=8.0)
    a = I.make_workload(spec, seed=3)
    b = I.make_workload(spec, seed=3)
    c = I.make_workload(spec, seed=4)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.w, b.w)
    assert np.array_equal(a.labels, b.labels)
    assert not np.array_equal(a.x, c.x)
    assert a.x.shape == (300, 40) and a.w.shape == (500, 40)
    assert a.x.dtype == np.uint16
    assert (a.labels == I.IGNORE_INDEX).sum() == 30
    v = a.labels[a.labels != I.IGNORE_INDEX]
    assert v.min() >= 0 and v.max() < 500


def test_recipe_statistics():
    spec = I.custom_spec("t", N=2048, H=256, V=3000, dtype="bf16", x_rms_rows=True,
                         n_scaled_w_rows=30, w_row_scale=8.0)
    wl = I.make_workload(spec, seed=0)
    x = wl.x_f32().astype(np.float64)
    rms = np.sqrt((x ** 2).mean(axis=1))
    assert np.allclose(rms, 1.0, atol=1e-2)
    w = wl.w_f32().astype(np.float64)
    row_std = w.std(axis=1)
    big = row_std > 0.08
    assert big.sum() == 30
    assert np.allclose(row_std[~big].mean(), 0.02, rtol=0.05)


def test_zipf_head_heavier_than_uniform():
    spec = I.custom_spec("t", N=20000, H=8, V=1000, dtype="fp32", labels="zipf")
    lab = I.make_labels(spec, 0)
    counts = np.bincount(lab, minlength=1000)
    # rank-1 mass of a finite Zipf(1.1) over 1000 ranks is about 0.16
    assert counts.max() / 20000 == pytest.approx(0.16, abs=0.03)


def test_configs_match_stated_shapes():
    c = I.CONFIGS
    assert (c["tiny"].N, c["tiny"].H, c["tiny"].V, c["tiny"].dtype) == (256, 256, 4096, "fp32")
    assert (c["llama3_n8192"].N, c["llama3_n8192"].n_ignore) == (8192, 410)
    assert (c["qwen25_n16384"].V, c["qwen25_n16384"].smoothing) == (152064, 0.1)
    assert (c["gemma2_n32768"].n_ignore, c["gemma2_n32768"].n_scaled_w_rows) == (1638, 2560)


def test_sft_prompt_spans():
    spec = I.custom_spec("t", N=1000, H=8, V=50, dtype="fp32", labels="sft", seq_len=250,
                         prompt_frac=(0.3, 0.6))
    lab = I.make_labels(spec, 0)
    for b in range(4):
        seq = lab[b * 250:(b + 1) * 250]
        ign = np.flatnonzero(seq == I.IGNORE_INDEX)
        # a contiguous prefix of 30-60% of the sequence is masked
        assert len(ign) == ign[-1] + 1 and 75 <= len(ign) <= 150
        assert np.all(seq[len(ign):] >= 0)


def test_peaked_targets_stand_out():
    spec = I.custom_spec("p", N=200, H=256, V=3000, dtype="bf16", x_align=3.0, n_ignore=10)
    wl = I.make_workload(spec, 0)
    x = wl.x_f32().astype(np.float64)
    w = wl.w_f32().astype(np.float64)
    z = x @ w.T
    valid = wl.labels != I.IGNORE_INDEX
    zy = z[np.flatnonzero(valid), wl.labels[valid]]
    assert np.median(zy) > 10.0 and np.std(z) < 2.0
