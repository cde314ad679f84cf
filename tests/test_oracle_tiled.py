"""Pins of the tiled-decode oracle (``oracle.wan_tiled``).

The blending is checked against closed forms written out here by hand (a
two-tile ramp, a four-tile corner), against a global field that any correctly
aligned convex blend must reproduce, and the whole tiled decode against the
untiled ``decode`` in the two cases where tiling must not change anything
(one tile covering the frame; tiles that do not overlap).
"""

import numpy as np
import pytest

import oracle
import wan_synth


def test_tile_origins_cover_the_axis():
    # 704 pixels (the 720p video's height), the default 256 / 192 tiles
    assert oracle.tile_origins(704, 256, 192) == [(0, 256), (192, 256), (384, 256), (576, 128)]
    # latents: 44 rows at tile 16, stride 12
    assert oracle.tile_origins(44, 16, 12) == [(0, 16), (12, 16), (24, 16), (36, 8)]
    assert oracle.tile_origins(5, 16, 12) == [(0, 5)]
    for n, t, s in [(1, 1, 1), (7, 3, 2), (13, 16, 12), (100, 9, 4), (64, 8, 8)]:
        o = oracle.tile_origins(n, t, s)
        kept = np.zeros(n, int)
        for a, size in o:
            assert 0 < size <= t and a + size <= n
            kept[a:a + min(s, size)] += 1  # the region each tile supplies
        assert (kept == 1).all()
    with pytest.raises(ValueError):
        oracle.tile_origins(10, 4, 5)


def _cut(field, H, W, tile, stride):
    """Tiles that are exact samples of one global field [..., H, W]."""
    rows = oracle.tile_origins(H, tile[0], stride[0])
    cols = oracle.tile_origins(W, tile[1], stride[1])
    return [[field[..., r:r + rh, c:c + cw].copy() for c, cw in cols] for r, rh in rows]


@pytest.mark.parametrize("H,W,tile,stride", [
    (96, 112, (64, 64), (48, 48)),     # short last row and a 16-pixel last column
    (80, 80, (64, 64), (16, 16)),      # overlap 48 > stride: blended rows are blended again
    (40, 72, (32, 48), (16, 48)),      # no overlap across columns
    (224, 224, (256, 256), (192, 192)),  # first tile cut by the frame edge
    (50, 30, (20, 12), (7, 5)),
])
def test_blend_reproduces_a_global_field(H, W, tile, stride):
    # weights summing to 1 at globally aligned pixels reproduce any field
    rng = np.random.default_rng(7)
    field = rng.standard_normal((2, 3, H, W))
    out = oracle.blend_tiles(_cut(field, H, W, tile, stride), H, W, *stride)
    np.testing.assert_allclose(out, field.astype(np.float32), rtol=0, atol=1e-6)


def test_blend_two_tile_ramp():
    # two tiles stacked vertically in 10 rows, constant 0 above and 1 below;
    # tile 8, stride 5: the lower tile holds rows 5..9, the overlap is rows
    # 5..7 (e = 3)
    assert oracle.tile_origins(10, 8, 5) == [(0, 8), (5, 5)]
    top, bot = np.zeros((1, 8, 4)), np.ones((1, 5, 4))
    out = oracle.blend_tiles([[top], [bot]], 10, 4, 5, 8)
    expect = np.array([0, 0, 0, 0, 0, 0, 1 / 3, 2 / 3, 1, 1], np.float32)
    np.testing.assert_allclose(out[0, :, 0], expect, rtol=0, atol=1e-7)
    assert (out == out[..., :1]).all()


def test_blend_four_tile_corner_closed_form():
    # constants a (top left), b (top right), c (bottom left), d (bottom right);
    # tile 10, stride 6, overlap e = 4.  Pixel (6 + y, 6 + x), y, x < 4, with
    # u = y / e, v = x / e.  The tile above (b) has already had its left
    # columns blended with a, the tile to the left (c) its top rows with a:
    #   after the vertical blend: (a (1 - v) + b v) (1 - u) + d u
    #   after the horizontal one: (a (1 - u) + c u) (1 - v) + that * v
    a, b, c, d = 0.3, -0.7, 0.9, 0.1
    tiles = [[np.full((10, 10), a), np.full((10, 6), b)], [np.full((6, 10), c), np.full((6, 6), d)]]
    out = oracle.blend_tiles(tiles, 12, 12, 6, 6)
    e = 4
    for y in range(e):
        for x in range(e):
            u, v = y / e, x / e
            vert = (a * (1 - v) + b * v) * (1 - u) + d * u
            expect = (a * (1 - u) + c * u) * (1 - v) + vert * v
            assert abs(out[6 + y, 6 + x] - expect) < 1e-6, (y, x)
    # away from the seams each tile keeps its own value
    assert out[0, 0] == np.float32(a) and out[0, 11] == np.float32(b)
    assert out[11, 0] == np.float32(c) and out[11, 11] == np.float32(d)


def test_blend_keeps_constants_and_range():
    rng = np.random.default_rng(3)
    tiles = _cut(np.full((1, 50, 70), 0.25), 50, 70, (20, 30), (12, 17))
    out = oracle.blend_tiles(tiles, 50, 70, 12, 17)
    np.testing.assert_allclose(out, 0.25, rtol=0, atol=1e-7)
    tiles = [[rng.uniform(-1, 1, t.shape) for t in row] for row in tiles]
    out = oracle.blend_tiles(tiles, 50, 70, 12, 17)
    assert out.min() >= -1 and out.max() <= 1


@pytest.fixture(scope="module")
def tiny():
    return wan_synth.make_weights(base=16, seed=0)


def test_one_tile_covering_the_frame_is_the_untiled_decode(tiny):
    z = wan_synth.make_latents((1, 48, 2, 3, 5), seed=1)
    ref = oracle.decode(z, tiny)
    for tile, stride in [((48, 80), (48, 80)), ((256, 256), (192, 192))]:
        np.testing.assert_array_equal(oracle.decode_tiled(z, tiny, tile=tile, stride=stride), ref)


def test_non_overlapping_tiles_are_independent_decodes(tiny):
    # stride == tile: each block of the output is the decode of its latent block
    z = wan_synth.make_latents((1, 48, 2, 5, 4), seed=2)
    out = oracle.decode_tiled(z, tiny, tile=(48, 32), stride=(48, 32))
    for r0 in (0, 3):
        for c0 in (0, 2):
            blk = oracle.decode(z[..., r0:r0 + 3, c0:c0 + 2], tiny)
            np.testing.assert_array_equal(out[..., 16 * r0:16 * r0 + blk.shape[-2], 16 * c0:16 * c0 + blk.shape[-1]],
                                          blk)


def test_tiled_decode_differs_from_untiled_and_stays_in_range(tiny):
    # overlapping tiles: each tile sees zero padding at its own edges, so the
    # result differs from the untiled decode (the pages report it for their
    # test model), while staying a convex blend of values in [-1, 1]
    z = wan_synth.make_latents((1, 48, 2, 6, 7), seed=1)
    ref = oracle.decode(z, tiny)
    out = oracle.decode_tiled(z, tiny, tile=(64, 64), stride=(48, 48))
    assert out.shape == ref.shape
    assert np.abs(out).max() <= 1.0
    diff = np.abs(out - ref).max()
    assert diff > 0


def test_tile_arguments_are_checked(tiny):
    z = wan_synth.make_latents((1, 48, 1, 2, 2), seed=1)
    for tile, stride in [((40, 32), (16, 16)), ((32, 32), (48, 16)), ((32, 32), (0, 16))]:
        with pytest.raises(ValueError):
            oracle.decode_tiled(z, tiny, tile=tile, stride=stride)


def test_wan21_tiles_use_eight_pixels_per_latent():
    # Wan2.1 decodes 8 pixels per latent: 16-pixel tiles are 2 latents; one
    # covering tile is the untiled decode, non-overlapping tiles are
    # independent block decodes
    w = wan_synth.make_weights(base=16, seed=0, variant="wan21")
    z = wan_synth.make_latents((1, 16, 2, 4, 4), seed=3)
    ref = oracle.decode(z, w)
    assert ref.shape[-2:] == (32, 32)
    np.testing.assert_array_equal(oracle.decode_tiled(z, w, tile=(32, 32), stride=(32, 32)), ref)
    out = oracle.decode_tiled(z, w, tile=(16, 32), stride=(16, 32))
    for r0 in (0, 2):
        np.testing.assert_array_equal(out[..., 8 * r0:8 * r0 + 16, :], oracle.decode(z[..., r0:r0 + 2, :], w))
