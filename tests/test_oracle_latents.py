"""Pins of the latent de-normalisation oracle (``oracle.wan_latents``).

Checked against an element-by-element loop, the identity statistics, the
standardisation it inverts, and the decode of latents de-normalised by hand.
"""

import numpy as np
import pytest

import oracle
import wan_synth


def _stats(seed=0, C=48):
    rng = np.random.default_rng(seed)
    return rng.uniform(-1, 1, C).astype(np.float32), rng.uniform(0.5, 3, C).astype(np.float32)


def test_denormalize_matches_an_elementwise_loop():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((2, 48, 2, 3, 4)).astype(np.float32)
    mean, std = _stats()
    got = oracle.denormalize_latents(z, mean, std)
    for b, c, t, y, x in np.ndindex(z.shape):
        want = float(z[b, c, t, y, x]) * float(std[c]) + float(mean[c])
        assert abs(got[b, c, t, y, x] - want) <= 1e-6 * max(1.0, abs(want))


def test_identity_statistics_and_inverse_of_standardisation():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((1, 48, 3, 2, 5)).astype(np.float32)
    np.testing.assert_array_equal(oracle.denormalize_latents(z, np.zeros(48), np.ones(48)), z)
    mean, std = _stats(3)
    x = oracle.denormalize_latents(z, mean, std)
    back = (x.astype(np.float64) - mean.reshape(1, 48, 1, 1, 1)) / std.reshape(1, 48, 1, 1, 1)
    np.testing.assert_allclose(back, z, rtol=0, atol=1e-5)
    # channel c depends only on mean[c], std[c]: change one channel's statistics
    mean2 = mean.copy()
    mean2[7] += 1.0
    d = oracle.denormalize_latents(z, mean2, std) - x
    assert np.all(d[:, 7] != 0) and np.all(np.delete(d, 7, axis=1) == 0)


def test_statistics_shape_checked():
    z = np.zeros((1, 48, 1, 1, 1), np.float32)
    with pytest.raises(ValueError):
        oracle.denormalize_latents(z, np.zeros(47), np.ones(48))


def test_decode_normalized_is_decode_of_denormalized_latents():
    w = wan_synth.make_weights(base=16, seed=0)
    z = wan_synth.make_latents((1, 48, 2, 2, 3), seed=4)
    mean, std = _stats(5)
    by_hand = (z.astype(np.float64) * std.reshape(1, 48, 1, 1, 1) + mean.reshape(1, 48, 1, 1, 1)).astype(np.float32)
    np.testing.assert_array_equal(oracle.decode_normalized(z, w, mean, std), oracle.decode(by_hand, w))
    np.testing.assert_array_equal(oracle.decode_normalized(z, w, mean, std, round_latents=oracle.round_bf16),
                                  oracle.decode(oracle.round_bf16(by_hand), w))
