"""Latent de-normalisation on the GPU (wan_vae_model_set_latent_stats)
against the oracle's decode of de-normalised latents."""

import numpy as np
import pytest
import torch

import oracle
import wan_synth
from tests.gpu_util import lib_ready, rounded, to_dev, weights_dev
from tests.parity_log import record

pytestmark = pytest.mark.gpu
TOL, PSNR_MIN = 4e-2, 40.0
TOL_F32 = 2e-3


@pytest.fixture(scope="module")
def wv():
    return lib_ready()


@pytest.fixture(scope="module")
def tiny():
    w = wan_synth.make_weights(base=16, seed=0)
    return w, weights_dev(w)


def _stats(seed=0):
    rng = np.random.default_rng(seed)
    return rng.uniform(-1, 1, 48).astype(np.float32), rng.uniform(0.5, 3, 48).astype(np.float32)


def _clip(wv, model, z, chunk=2):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    v = st.decode_clip(to_dev(z), out_dtype=torch.float32)
    st.sync_status()
    return v.cpu().numpy()


def test_denormalized_decode_bf16(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 3, 4, 4), seed=11)
    mean, std = _stats()
    model = wv.Model(wd, dtype=torch.bfloat16)
    model.set_latent_stats(mean, std)
    got = _clip(wv, model, z)
    ref = oracle.decode_normalized(z, rounded(w), mean, std, round_latents=oracle.round_bf16)
    err, p = float(np.abs(got - ref).max()), oracle.psnr(got, ref)
    record("tiny bf16, de-normalised latents", err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)


def test_denormalized_decode_fp32(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=12)
    mean, std = _stats(1)
    model = wv.Model(wd, dtype=torch.float32)
    model.set_latent_stats(mean, std)
    got = _clip(wv, model, z)
    err = float(np.abs(got - oracle.decode_normalized(z, w, mean, std)).max())
    record("tiny fp32, de-normalised latents", err, None)
    assert err <= TOL_F32, err


def test_identity_statistics_and_switching_off(wv, tiny):
    _, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=13)
    model = wv.Model(wd, dtype=torch.bfloat16)
    plain = _clip(wv, model, z)
    model.set_latent_stats(np.zeros(48), np.ones(48))   # z * 1 + 0 is z exactly
    np.testing.assert_array_equal(_clip(wv, model, z), plain)
    model.set_latent_stats(*_stats(2))
    assert not np.array_equal(_clip(wv, model, z), plain)
    model.set_latent_stats(None, None)
    np.testing.assert_array_equal(_clip(wv, model, z), plain)


def test_denormalized_tiled_decode(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 6, 7), seed=14)
    mean, std = _stats(3)
    model = wv.Model(wd, dtype=torch.bfloat16)
    model.set_latent_stats(mean, std)
    got = model.decode_tiled(to_dev(z), tile=(64, 64), stride=(48, 48)).float().cpu().numpy()
    x = oracle.round_bf16(oracle.denormalize_latents(z, mean, std))
    ref = oracle.decode_tiled(x, rounded(w), tile=(64, 64), stride=(48, 48))
    err, p = float(np.abs(got - ref).max()), oracle.psnr(got, ref)
    record("tiled tiny bf16, de-normalised latents", err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)


def test_statistics_arguments(wv, tiny):
    _, wd = tiny
    model = wv.Model(wd, dtype=torch.bfloat16)
    with pytest.raises(wv.WanError):
        model.set_latent_stats(np.zeros(47), np.ones(47))
    with pytest.raises(wv.WanError):
        model.set_latent_stats(np.zeros(48), np.full(48, np.inf))
    with pytest.raises(ValueError):
        model.set_latent_stats(np.zeros(48), np.ones(47))
