"""The seeded input recipes: determinism, shapes and the stated distributions."""
import numpy as np

import synth


def test_determinism_and_shapes():
    a = synth.kv_tensor(1)
    b = synth.kv_tensor(1)
    assert a.dtype == np.float16 and a.shape == (4096, 64)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(synth.kv_tensor(5, 0, rows=100), synth.kv_tensor(5, 1, rows=100))


def test_channel_scaled_recipe():
    x = synth.kv_tensor(2, 0).astype(np.float32).reshape(12, 12, 1024, 64)
    sd = x.std(axis=2)                       # per (layer, head, channel)
    top = np.sort(sd, axis=2)
    # one outlier channel per (layer, head), 20x a log-uniform [0.5, 8] scale
    assert np.all(top[..., -1] > 9.0)
    assert np.all(top[..., -2] < 9.0) and np.all(top[..., 0] > 0.4)


def test_token_lognormal_recipe_small_prefix():
    w = synth.WORKLOADS[4]
    assert w.rows == 32 * 8 * 32768 and w.d == 128
    r = synth.rng(4, synth.STREAM_K)
    s = r.lognormal(0.0, 0.5, size=(8, 32768, 1))
    assert abs(np.log(s).std() - 0.5) < 0.01


def test_gather_indices():
    i = synth.gather_indices(2, 0, 147456, 65536)
    assert i.dtype == np.int64 and i.min() >= 0 and i.max() < 147456
    p = synth.token_positions(4, 32768, 3277)
    assert np.unique(p).size == 3277
