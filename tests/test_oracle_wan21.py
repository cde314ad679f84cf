"""Pins of the oracle's Wan2.1 decode (z_dim 16, 8x spatial).

The parts are the TI2V-5B decode's, pinned in ``test_oracle_pins.py``.  The
composition is pinned by the frame counts and sizes, frame loop = whole
sequence, causality, batch independence, a separately written whole-sequence
torch composition, and the Wan2.1-specific wiring: resamplers that halve the
channels and no DupUp3D shortcut (zeroing an up block's resampler weights
must zero what that block hands on, which DupUp3D would not).
"""

import numpy as np
import pytest

import oracle
import wan_synth


@pytest.fixture(scope="module")
def w21():
    return wan_synth.make_weights(base=16, seed=0, variant="wan21")


def test_weight_table_is_the_wan21_layout(w21):
    assert oracle.is_wan21(w21)
    assert not oracle.is_wan21(wan_synth.make_weights(base=16, seed=0))
    assert w21["post_quant_conv.weight"].shape == (16, 16, 1, 1, 1)
    assert w21["decoder.conv_in.weight"].shape == (64, 16, 3, 3, 3)
    assert w21["decoder.up_blocks.0.upsamplers.0.resample.1.weight"].shape == (32, 64, 3, 3)
    assert w21["decoder.up_blocks.1.resnets.0.conv_shortcut.weight"].shape == (64, 32, 1, 1, 1)
    assert w21["decoder.up_blocks.2.upsamplers.0.resample.1.weight"].shape == (16, 32, 3, 3)
    assert "decoder.up_blocks.2.upsamplers.0.time_conv.weight" not in w21
    assert w21["decoder.conv_out.weight"].shape == (3, 16, 3, 3, 3)


@pytest.mark.parametrize("T", [1, 2, 3])
def test_frame_count_and_size(w21, T):
    z = wan_synth.make_latents((1, 16, T, 3, 5), seed=2)
    v = oracle.decode(z, w21)
    assert v.shape == (1, 3, 4 * T - 3, 24, 40)
    assert np.isfinite(v).all() and np.abs(v).max() <= 1


def test_frame_loop_equals_whole_sequence(w21):
    z = wan_synth.make_latents((1, 16, 3, 4, 4), seed=1)
    _, f1 = oracle.decode(z, w21, chunk=1, return_preclamp=True)
    _, f2 = oracle.decode_whole(z, w21, return_preclamp=True)
    assert np.abs(f1 - f2).max() <= 1e-4 * np.abs(f2).max()


def test_causality(w21):
    z = wan_synth.make_latents((1, 16, 3, 3, 3), seed=3)
    base = oracle.decode(z, w21)
    z2 = z.copy()
    z2[:, :, 2] += 1.0
    other = oracle.decode(z2, w21)
    np.testing.assert_array_equal(base[:, :, :5], other[:, :, :5])   # frames of latents 0, 1
    assert not np.array_equal(base[:, :, 5:], other[:, :, 5:])


def test_batch_independence(w21):
    z = wan_synth.make_latents((2, 16, 2, 3, 3), seed=4)
    both = oracle.decode(z, w21)
    for b in range(2):
        np.testing.assert_allclose(both[b:b + 1], oracle.decode(z[b:b + 1], w21), rtol=0, atol=2e-6)


def test_resampler_is_the_only_path_between_levels(w21):
    # with up block 2's resampler zeroed, level D sees zeros; a DupUp3D
    # shortcut (TI2V-5B) would still carry the block input through
    w = dict(w21)
    w["decoder.up_blocks.2.upsamplers.0.resample.1.weight"] = np.zeros((16, 32, 3, 3), np.float32)
    w["decoder.up_blocks.2.upsamplers.0.resample.1.bias"] = np.zeros(16, np.float32)
    z1 = wan_synth.make_latents((1, 16, 2, 3, 3), seed=5)
    z2 = wan_synth.make_latents((1, 16, 2, 3, 3), seed=6)
    np.testing.assert_array_equal(oracle.decode(z1, w), oracle.decode(z2, w))


def test_oracle_vs_independent_torch_composition(w21):
    from tests.torch_composition import decode_whole_torch
    z = wan_synth.make_latents((1, 16, 3, 4, 4), seed=1)
    _, pre = oracle.decode(z, w21, return_preclamp=True)
    want = decode_whole_torch(z, w21)
    assert want.shape == pre.shape == (1, 3, 9, 32, 32)
    assert np.abs(pre - want).max() <= 1e-4 * np.abs(want).max()
