"""The seeded generators draw what the workload recipes state."""
import numpy as np

import synth


def test_stream_is_deterministic_and_split():
    a = synth.u64(0, "X", 1000)
    assert np.array_equal(a, synth.u64(0, "X", 1000))
    assert np.array_equal(a[10:20], synth.u64(0, "X", 10, offset=10))
    assert not np.array_equal(a, synth.u64(0, "Y", 1000))
    assert not np.array_equal(a, synth.u64(1, "X", 1000))


def test_splitmix64_published_first_outputs():
    # SplitMix64 seeded with state 0 yields, as its first outputs, mix(GAMMA),
    # mix(2*GAMMA): 0xE220A8397B1DCDAF and 0x6E789E6AA1B965F4.
    g = synth._GAMMA
    with np.errstate(over="ignore"):
        z = np.array([g, g * np.uint64(2)], dtype=np.uint64)
    out = synth._mix(z)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_normal_moments():
    z = synth.normal(0, "moments", 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def test_code_distributions():
    q4 = synth.codes(synth.Q4_0, 256, 1024, 0, "W")
    assert q4.min() == 0 and q4.max() == 15
    assert np.all(np.abs(np.bincount(q4.ravel(), minlength=16) / q4.size - 1 / 16) < 0.002)
    q8 = synth.codes(synth.Q8_0, 256, 1024, 0, "W")
    assert q8.min() >= -127 and q8.max() <= 127 and abs(q8.std() - 40) < 0.5
    q2 = synth.codes(synth.Q2_0, 256, 1024, 0, "W")
    frac = np.bincount(q2.ravel(), minlength=4) / q2.size
    assert abs(frac[3] - 0.01) < 0.002
    assert np.allclose(frac[:3], np.array([0.3, 0.4, 0.3]) * 0.99, atol=0.005)


def test_scales_are_nonnegative_fp16():
    d = synth.scales(synth.Q4_0, 64, 256, 0, "W")
    assert d.dtype == np.float16 and d.shape == (64, 8) and np.all(d >= 0)


def test_pack_shapes():
    for c in synth.CODECS:
        K = 1024
        W = synth.weights(c, 8, K, 0)
        assert W.shape == (8, synth.row_bytes(c, K)) and W.dtype == np.uint8


def test_mlx4_biases_follow_recipe():
    d = synth.scales(synth.MLX4, 64, 1024, 0, "W")
    b = synth.biases(synth.MLX4, 64, 1024, 0, "W", d)
    assert b.dtype == np.float16 and b.shape == (64, 32)
    big = d.astype(np.float64) > 1e-3
    ratio = -(b.astype(np.float64) / d.astype(np.float64))[big]
    assert abs(ratio.mean() - 7.5) < 0.05 and abs(ratio.std() - 0.5) < 0.05
    assert synth.biases(synth.Q4_0, 64, 1024, 0, "W", d) is None


def test_mlx4_planar_and_block_layouts():
    N, K = 4, 64
    q = synth.codes(synth.MLX4, N, K, 0, "W")
    d = synth.scales(synth.MLX4, N, K, 0, "W")
    b = synth.biases(synth.MLX4, N, K, 0, "W", d)
    words, s, bb = synth.planar(q, d, b)
    assert words.dtype == np.uint32 and words.shape == (N, K // 8)
    # code k sits at bits 4 (k % 8) of word k // 8
    for k in (0, 1, 7, 8, 37, 63):
        assert np.array_equal((words[:, k // 8] >> np.uint32(4 * (k % 8))) & np.uint32(15), q[:, k])
    W = synth.pack(synth.MLX4, q, d, b).reshape(N, K // 32, 20)
    assert np.array_equal(W[:, :, 0:2].copy().view("<u2")[..., 0], d.view("<u2"))
    assert np.array_equal(W[:, :, 2:4].copy().view("<u2")[..., 0], b.view("<u2"))
    # the 16 code bytes of a block are the planar words' bytes of that group
    assert np.array_equal(W[:, :, 4:].reshape(N, -1), words.view(np.uint8).reshape(N, -1))


def test_kv_cache_layouts():
    K = synth.kv_cache(synth.KV_F16, 2, 10, 64, 0, "K")
    assert K.dtype == np.float16 and K.shape == (2, 10, 64)
    Kq = synth.kv_cache(synth.Q8_0, 2, 10, 128, 0, "K")
    assert Kq.dtype == np.uint8 and Kq.shape == (2, 10, 4 * 34)
    assert synth.queries(4, 3, 64, 0).shape == (4, 3, 64)
