"""Tiled decode on the GPU (wan_vae_decode_tiled) against the tiled-decode
oracle, and against the untiled GPU decode where tiling must change nothing.

Geometries cover mixed tile sizes with a 16-pixel last column, an overlap
larger than the stride (rows blended twice), no overlap along one axis, a
single tile covering the frame, a batch of two, and several tile batches.
"""

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


GEOMETRIES = [
    # latents, tile, stride (pixels)
    ((1, 48, 2, 6, 7), (64, 64), (48, 48)),     # tiles 4/3 x 4/4/1 latents
    ((1, 48, 1, 5, 5), (64, 64), (16, 16)),     # 5 x 5 tiles, overlap 48 > stride
    ((2, 48, 2, 3, 5), (32, 48), (16, 48)),     # B = 2; columns do not overlap
    ((1, 48, 3, 4, 4), (256, 256), (192, 192)),  # one tile covers the frame
]


@pytest.mark.parametrize("shape,tile,stride", GEOMETRIES)
def test_tiled_tiny_bf16(wv, tiny, shape, tile, stride):
    w, wd = tiny
    z = wan_synth.make_latents(shape, seed=1)
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = model.decode_tiled(to_dev(z), tile=tile, stride=stride, max_chunk=2).float().cpu().numpy()
    ref = oracle.decode_tiled(oracle.round_bf16(z), rounded(w), tile=tile, stride=stride)
    err = float(np.abs(got - ref).max())
    p = oracle.psnr(got, ref)
    record(f"tiled tiny bf16 {shape} tile {tile} stride {stride}", err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)


def test_tiled_tiny_fp32(wv, tiny):
    w, wd = tiny
    shape, tile, stride = GEOMETRIES[0]
    z = wan_synth.make_latents(shape, seed=3)
    model = wv.Model(wd, dtype=torch.float32)
    got = model.decode_tiled(to_dev(z), tile=tile, stride=stride, out_dtype=torch.float32).cpu().numpy()
    ref = oracle.decode_tiled(z, w, tile=tile, stride=stride)
    err = float(np.abs(got - ref).max())
    record(f"tiled tiny fp32 {shape} tile {tile} stride {stride}", err, oracle.psnr(got, ref))
    assert err <= TOL_F32, err


def _untiled(wv, model, z, chunk):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    v = st.decode_clip(z, out_dtype=torch.float32)
    st.sync_status()
    return v


def test_single_tile_equals_untiled_decode(wv, tiny):
    _, wd = tiny
    z = to_dev(wan_synth.make_latents((1, 48, 3, 4, 5), seed=4))
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = model.decode_tiled(z, tile=(256, 256), stride=(192, 192), out_dtype=torch.float32, max_chunk=2)
    assert torch.equal(got, _untiled(wv, model, z, 2))


def test_non_overlapping_tiles_equal_block_decodes(wv, tiny):
    _, wd = tiny
    z = to_dev(wan_synth.make_latents((1, 48, 2, 5, 4), seed=2))
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = model.decode_tiled(z, tile=(48, 32), stride=(48, 32), out_dtype=torch.float32)
    for r0 in (0, 3):
        for c0 in (0, 2):
            blk = _untiled(wv, model, z[..., r0:r0 + 3, c0:c0 + 2].contiguous(), 4)
            assert torch.equal(got[..., 16 * r0:16 * r0 + blk.shape[-2], 16 * c0:16 * c0 + blk.shape[-1]], blk)


def test_tile_batching_does_not_change_the_result(wv, tiny):
    # the same tiles decoded one per batch, two per batch, or all together
    _, wd = tiny
    z = to_dev(wan_synth.make_latents((1, 48, 2, 6, 7), seed=5))
    model = wv.Model(wd, dtype=torch.bfloat16)
    runs = [model.decode_tiled(z, tile=(64, 64), stride=(48, 48), out_dtype=torch.float32, tile_batch=tb)
            for tb in (0, 1, 2)]
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])


def test_tiled_bf16_latents_and_output(wv, tiny):
    # bf16 latents go through the gather as 16-bit words
    _, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 6, 7), seed=6)
    model = wv.Model(wd, dtype=torch.bfloat16)
    a = model.decode_tiled(to_dev(oracle.round_bf16(z)), tile=(64, 64), stride=(48, 48), out_dtype=torch.float32)
    b = model.decode_tiled(to_dev(z, torch.bfloat16), tile=(64, 64), stride=(48, 48), out_dtype=torch.bfloat16)
    assert torch.equal(a.to(torch.bfloat16), b)


def test_tiled_full_width(wv):
    w = wan_synth.make_weights(base=256, seed=0)
    z = wan_synth.make_latents((1, 48, 2, 6, 6), seed=1)
    model = wv.Model(weights_dev(w), dtype=torch.bfloat16)
    got = model.decode_tiled(to_dev(z), tile=(64, 64), stride=(48, 48)).float().cpu().numpy()
    ref = oracle.decode_tiled(oracle.round_bf16(z), rounded(w), tile=(64, 64), stride=(48, 48))
    err = float(np.abs(got - ref).max())
    p = oracle.psnr(got, ref)
    record("tiled full-width bf16 [1,48,2,6,6] tile 64 stride 48", err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)
