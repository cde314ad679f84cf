"""Full-size parity: the 720p, portrait and 480p batch-2 workloads decoded in
the benchmark's launch configuration (bf16, chunks of 4 latent frames).

The oracle computes the first output frame of each (a decode of latent frame
0 alone: output frame 0 depends on nothing else, by the causal structure of
section "Causal caches"); the rest of each clip is checked through
properties that hold at any size: the decode of a prefix of the latents
reproduces the clip's leading frames bit for bit, and every value is finite
and inside [-1, 1].
"""

import numpy as np
import pytest
import torch

import oracle
import wan_synth
from tests.gpu_util import lib_ready, rounded, to_dev, weights_dev
from tests.parity_log import record

pytestmark = pytest.mark.gpu
CHUNK = 4


@pytest.fixture(scope="module")
def full():
    wv = lib_ready()
    w = wan_synth.make_weights(base=256, seed=0)
    model = wv.Model(weights_dev(w), dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return wv, w, model


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


@pytest.mark.parametrize("name", ["720p", "portrait", "480p_b2"])
def test_full_size_first_frame_and_prefix(full, name):
    wv, w, model = full
    cfg = wan_synth.CONFIGS[name]
    z = wan_synth.make_latents(cfg["latents"], cfg["latent_seed"])
    video = _decode(wv, model, z)
    B, _, T, h, wl = z.shape
    assert video.shape == (B, 3, 4 * T - 3, 16 * h, 16 * wl)
    assert np.isfinite(video).all() and np.abs(video).max() <= 1.0
    # frame 0 against the oracle (bf16-rounded inputs, fp32 arithmetic)
    ref0 = oracle.decode(oracle.round_bf16(z[:, :, :1]), rounded(w))
    got0 = video[:, :, :1]
    err = float(np.abs(got0 - ref0).max())
    p = oracle.psnr(got0, ref0)
    record(f"{name} frame 0 (bf16)", err, p)
    assert err <= 4e-2 and p >= 40.0, (err, p)
    # prefix: latent frames 0..4 give the clip's first 17 frames exactly
    pre = _decode(wv, model, np.ascontiguousarray(z[:, :, :5]))
    np.testing.assert_array_equal(pre, video[:, :, :17])
