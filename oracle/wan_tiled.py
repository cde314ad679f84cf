"""Tiled decode: the decode of overlapping latent tiles, blended at the seams
(CPU oracle; test infrastructure only, the CUDA path never imports it).

Source: the page "[Feature] Implement tiled VAE encoding/decoding for Wan
model. #11414" (diffusers pull request).  It fixes the interface: tiling is
opt-in, a tile has a sample-space height and width, tiles are placed at a
sample-space stride, the defaults are 256 (tile) and 192 (stride), and the
tiled result may differ from the untiled one (a max difference of about 0.4
on a random-weight test model, with the arrays' mean magnitude under 0.01).
It does not print the blending.  The reading taken here, the plainest one
consistent with "tiles overlap by tile - stride and are blended":

* Tile origins.  Along each spatial axis of N pixels, tiles start at 0,
  stride, 2*stride, ... (every start < N) and cover min(tile, N - start)
  pixels.  In latents (P = 16 video pixels per latent; P = 8 for the Wan2.1
  decoder) that is tile/P latents at a stride of stride/P latents; both
  sizes must be multiples of 16 pixels.
* Each tile is decoded on its own by ``decode`` (all frames, its own causal
  caches, unpatchify and clamp included), as if it were the whole latent.
* Blending, in raster order over the tiles, in place: tile (i, j) first
  cross-fades its top rows with the rows of the (already blended) tile above
  that cover the same pixels, then its left columns with the columns of the
  (already blended) tile to its left that cover the same pixels.  Over an
  overlap of e pixels, local row (column) k < e of the later tile becomes
  earlier * (e - k) / e + later * k / e.  e is the number of pixels the two
  tiles share, which is tile - stride wherever the earlier tile is not cut
  by the frame edge.
* Assembly: tile (i, j) supplies the pixels from its origin up to the next
  tile's origin (its first `stride` rows and columns, or fewer at the frame
  edge).  These regions partition the frame.

The blend weights sum to 1, so every output pixel is a convex combination of
decoded values and stays in [-1, 1].
"""

from __future__ import annotations

import numpy as np

from .wan_decode import decode, is_wan21

# 8x spatial upsampling in the decoder, then the 2x2 unpatchify (TI2V-5B; the
# Wan2.1 decoder has no unpatchify: 8).  Tile sizes are multiples of 16 for both.
PIXELS_PER_LATENT = 16


def tile_origins(n: int, tile: int, stride: int) -> list[tuple[int, int]]:
    """(start, size) of the tiles along one axis of n pixels (or latents)."""
    if tile <= 0 or stride <= 0 or stride > tile:
        raise ValueError(f"need 0 < stride <= tile, got tile={tile} stride={stride}")
    return [(s, min(tile, n - s)) for s in range(0, n, stride)]


def blend_tiles(tiles, H: int, W: int, stride_h: int, stride_w: int) -> np.ndarray:
    """Blend decoded tiles into one [..., H, W] frame stack.

    ``tiles[i][j]`` is the decoded tile whose origin is (i * stride_h,
    j * stride_w), an array [..., Hij, Wij].  Computed in fp64, returned fp32.
    """
    t = [[np.array(x, dtype=np.float64) for x in row] for row in tiles]
    lead = t[0][0].shape[:-2]
    out = np.zeros(lead + (H, W), np.float64)
    for i, row in enumerate(t):
        for j, b in enumerate(row):
            if i > 0:  # top rows against the tile above
                a = t[i - 1][j]
                e = min(a.shape[-2] - stride_h, b.shape[-2])
                for k in range(e):
                    b[..., k, :] = a[..., k + stride_h, :] * ((e - k) / e) + b[..., k, :] * (k / e)
            if j > 0:  # then left columns against the tile to the left
                a = row[j - 1]
                e = min(a.shape[-1] - stride_w, b.shape[-1])
                for k in range(e):
                    b[..., :, k] = a[..., :, k + stride_w] * ((e - k) / e) + b[..., :, k] * (k / e)
            y0, x0 = i * stride_h, j * stride_w
            kh, kw = min(stride_h, b.shape[-2]), min(stride_w, b.shape[-1])
            out[..., y0:y0 + kh, x0:x0 + kw] = b[..., :kh, :kw]
    return out.astype(np.float32)


def decode_tiled(z, weights, tile=(256, 256), stride=(192, 192), chunk: int = 1) -> np.ndarray:
    """Tiled decode of z [B, 48, T, h, w] -> video [B, 3, 4T-3, 16h, 16w]
    (Wan2.1: z [B, 16, T, h, w] -> [B, 3, 4T-3, 8h, 8w]).

    ``tile`` and ``stride`` are (height, width) in video pixels, multiples of
    16.  Each latent tile goes through ``decode`` (frame loop of ``chunk``
    latent frames); the decoded tiles are blended by ``blend_tiles``.
    """
    z = np.asarray(z, np.float32)
    _, _, _, h, w = z.shape
    for v in (*tile, *stride):
        if v <= 0 or v % PIXELS_PER_LATENT:
            raise ValueError(f"tile and stride must be positive multiples of {PIXELS_PER_LATENT} pixels, "
                             f"got {tile}, {stride}")
    P = 8 if is_wan21(weights) else PIXELS_PER_LATENT  # video pixels per latent
    rows = tile_origins(h, tile[0] // P, stride[0] // P)
    cols = tile_origins(w, tile[1] // P, stride[1] // P)
    tiles = [[decode(z[..., r0:r0 + rh, c0:c0 + cw], weights, chunk=chunk) for c0, cw in cols] for r0, rh in rows]
    return blend_tiles(tiles, P * h, P * w, stride[0], stride[1])
