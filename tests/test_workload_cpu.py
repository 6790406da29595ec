"""The seeded input generators shared by the GPU path and the oracle (no layer
arithmetic): determinism and the distributions the workloads specify."""
import numpy as np

import workload as W


def test_route_noise_is_seeded_per_step_and_layer():
    a = W.route_noise(2, 3, 5, 128, 1.5)
    assert a.dtype == np.float32 and a.shape == (128,)
    assert np.array_equal(a, W.route_noise(2, 3, 5, 128, 1.5))
    assert not np.array_equal(a, W.route_noise(2, 3, 6, 128, 1.5))   # another step
    assert not np.array_equal(a, W.route_noise(2, 4, 5, 128, 1.5))   # another layer
    assert not np.array_equal(a, W.route_noise(3, 3, 5, 128, 1.5))   # another seed
    # values are bf16 numbers (the low 16 bits of the fp32 pattern are zero)
    assert not (a.view(np.uint32) & 0xffff).any()


def test_route_noise_moments():
    v = np.concatenate([W.route_noise(2, l, t, 128, 1.5) for l in range(8) for t in range(64)]).astype(np.float64)
    assert abs(v.mean()) < 0.05
    assert abs(v.std() - 1.5) < 0.05


def test_zipf_bias_is_alpha_log_popularity_over_a_permutation():
    E, s, alpha = 128, 1.1, 0.35
    bias, perm = W.zipf_bias(2, 0, E, s, alpha)
    assert sorted(perm.tolist()) == list(range(E))
    p = np.arange(1, E + 1, dtype=np.float64) ** -s
    p /= p.sum()
    assert np.allclose(bias[perm], alpha * np.log(p), rtol=1e-5, atol=1e-5)


def test_repeat_coin_is_fair_and_seeded():
    flips = [W.coin(2, l, t) for l in range(8) for t in range(256)]
    assert flips == [W.coin(2, l, t) for l in range(8) for t in range(256)]
    assert 0.45 < np.mean(flips) < 0.55
