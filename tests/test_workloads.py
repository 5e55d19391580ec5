"""The seeded input generator: determinism, bf16 rounding, masks, lengths."""
import numpy as np

import workloads as W


def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties go to the even (1.0)
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 3.140625, 1e-3],
                 np.float32)
    got = W.bf16_bits_to_f64(W.f32_to_bf16_bits(x))
    want = [1.0, 1.0, 1.0 + 2 * 2.0 ** -7, -2.5, 3.140625]
    np.testing.assert_array_equal(got[:5], want)
    # the nearest bf16 of 1e-3 is within half an ulp (2^-8 relative)
    assert abs(got[5] - 1e-3) <= 1e-3 * 2.0 ** -8


def test_bf16_widening_is_exact_roundtrip():
    rng = np.random.default_rng(0)
    bits = W.f32_to_bf16_bits(rng.standard_normal(1000).astype(np.float32))
    back = W.f32_to_bf16_bits(W.bf16_bits_to_f64(bits).astype(np.float32))
    np.testing.assert_array_equal(bits, back)


def test_generation_is_deterministic():
    a = W.make("tiny")
    b = W.make("tiny")
    for n in ("q", "k", "v", "do"):
        np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
    c = W.make("tiny", seed=99)
    assert not np.array_equal(a.q, c.q)


def test_bert_lengths_and_scale():
    w = W.make("bert")
    assert w.kv_len.dtype == np.int32 and w.kv_len.shape == (16,)
    assert w.kv_len.min() >= 256 and w.kv_len.max() <= 512
    # Q scaled by 0.5: std close to 0.5
    assert abs(np.std(w.f64("q")) - 0.5) < 0.01


def test_peaky_keys_gpt2_4k_shape():
    w = W.make("gpt2_4k", B=1, H=2)
    k = w.f64("k")
    # 41 rows per head hold |k| values far beyond a normal draw's range
    big = (np.abs(k).max(axis=-1) > 8.0).sum(axis=-1)
    assert big.shape == (1, 2)
    assert np.all(big <= 41) and np.all(big >= 30)


def test_sparse_mask_band_and_density():
    rng = np.random.default_rng(5)
    m = W.make_block_mask(rng, 512, 0.05, 1)
    assert m.shape == (512, 512) and m.dtype == np.uint8
    assert int(m.sum()) == 13107
    i = np.arange(512)
    assert np.all(m[i, i] == 1) and np.all(m[i[:-1], i[:-1] + 1] == 1)
    assert np.all(m[i[1:], i[1:] - 1] == 1)


def test_sampling_helpers():
    rng = np.random.default_rng(1)
    rows = W.sample_rows(rng, 2, 3, 100, 10)
    assert rows.shape == (60,) and len(np.unique(rows)) == 60
    assert rows.min() >= 0 and rows.max() < 600
    keys = W.sample_key_tiles(rng, 1, 2, 300, 2)
    # tiles of 128 rows; the last tile of N=300 holds 44 rows
    for bh in range(2):
        n = int(((keys >= bh * 300) & (keys < (bh + 1) * 300)).sum())
        assert n in (128 * 2, 128 + 44)
    assert np.all(np.diff(keys) > 0)
