"""Full-size parity: the 720p, portrait and 480p batch-2 workloads (and the
Wan2.1 VAE's 720p workload) decoded at full spatial size, bf16, against the
CPU oracle.

The oracle decodes (frame loop, bf16-rounded inputs, fp32 arithmetic) run in
background worker processes (``tests.oracle_jobs``) while the GPU decodes run:

- 720p and portrait: latent frames 0-1, i.e. output frames 0-4.  The GPU
  decodes them three ways: one latent frame per chunk (the second chunk is a
  steady-state chunk that reads every causal conv's two history frames from
  its ring at full size, across the chunk boundary: section "Causal caches"
  of the page "wan22_vae_decode/reference.py"); both latent frames as one
  chunk (the first-chunk rule of section "The first latent frame yields one
  frame" at full size); and frames 0-4 of the whole clip decoded in the
  benchmark's launch configuration (chunks of 4 latent frames).
- 480p batch 2 and Wan2.1 720p (attention over 90 x 160 = 14,400 positions):
  output frame 0.

Each frame is compared element by element: max |diff| <= 4e-2 and PSNR >= 40
dB.  The rest of each clip is checked through properties that hold at any
size: the decode of a prefix of the latents reproduces the clip's leading
frames bit for bit, and every value is finite and inside [-1, 1].
"""

import numpy as np
import pytest
import torch

import oracle
import wan_synth
from tests import oracle_jobs
from tests.gpu_util import lib_ready, to_dev, weights_dev
from tests.parity_log import record

pytestmark = pytest.mark.gpu
CHUNK = 4
TOL, PSNR_MIN = 4e-2, 40.0


@pytest.fixture(scope="module")
def models():
    wv = lib_ready()
    cache = {}

    def get(variant):
        if variant not in cache:
            base = 96 if variant == "wan21" else 256
            w = wan_synth.make_weights(base=base, seed=0, variant=variant)
            cache[variant] = wv.Model(weights_dev(w), dtype=torch.bfloat16)
            torch.cuda.synchronize()
        return cache[variant]

    return wv, get


def _decode(wv, model, z, chunk=CHUNK):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    out = st.decode_clip(to_dev(z), out_dtype=torch.bfloat16)
    st.sync_status()
    v = out.float().cpu().numpy()
    st.close()
    del out
    torch.cuda.empty_cache()
    return v


def _compare(case, got, ref):
    """Per output frame: max |diff| and PSNR against the oracle."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    for f in range(ref.shape[2]):
        err = float(np.abs(got[:, :, f] - ref[:, :, f]).max())
        p = oracle.psnr(got[:, :, f], ref[:, :, f])
        record(f"{case} frame {f} (bf16)", err, p)
        assert err <= TOL and p >= PSNR_MIN, (case, f, err, p)


@pytest.mark.parametrize("name", ["720p", "portrait"])
def test_full_size_first_two_latent_frames(models, name):
    wv, get = models
    model = get("ti2v")
    cfg = wan_synth.CONFIGS[name]
    z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
    z2 = np.ascontiguousarray(z[:, :, :2])
    one = _decode(wv, model, z2, chunk=1)        # chunk 1 reads full-size ring history
    both = _decode(wv, model, z2, chunk=2)       # one two-frame first chunk
    video = _decode(wv, model, z)                # the benchmark's configuration
    B, _, T, h, wl = z.shape
    assert video.shape == (B, 3, 4 * T - 3, 16 * h, 16 * wl)
    assert np.isfinite(video).all() and np.abs(video).max() <= 1.0
    ref = oracle_jobs.result(name, 2)
    _compare(f"{name} chunks of 1", one, ref)
    _compare(f"{name} one chunk of 2", both, ref)
    _compare(f"{name} clip, chunks of {CHUNK}", video[:, :, :5], ref)
    # prefix: latent frames 0..4 give the clip's first 17 frames exactly
    pre = _decode(wv, model, np.ascontiguousarray(z[:, :, :5]))
    np.testing.assert_array_equal(pre, video[:, :, :17])


def test_full_size_480p_batch2(models):
    wv, get = models
    model = get("ti2v")
    cfg = wan_synth.CONFIGS["480p_b2"]
    z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
    video = _decode(wv, model, z)
    B, _, T, h, wl = z.shape
    assert video.shape == (B, 3, 4 * T - 3, 16 * h, 16 * wl)
    assert np.isfinite(video).all() and np.abs(video).max() <= 1.0
    _compare("480p_b2 clip", video[:, :, :1], oracle_jobs.result("480p_b2", 1))
    pre = _decode(wv, model, np.ascontiguousarray(z[:, :, :5]))
    np.testing.assert_array_equal(pre, video[:, :, :17])


def test_full_size_wan21_720p_first_frame(models):
    """The Wan2.1 decode of 90 x 160 latents: its attention runs over 14,400
    positions per frame (page "Fix the Wan VAE attention block")."""
    wv, get = models
    model = get("wan21")
    cfg = wan_synth.CONFIGS["wan21_720p"]
    z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
    z1 = np.ascontiguousarray(z[:, :, :1])
    got = _decode(wv, model, z1)
    assert got.shape == (1, 3, 1, 720, 1280)
    _compare("wan21_720p", got, oracle_jobs.result("wan21_720p", 1))
