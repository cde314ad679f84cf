"""CPU oracle of the Wan2.2-TI2V-5B VAE decode (test infrastructure only).

A plain, slow NumPy implementation of what the decode computes, written from
the page "wan22_vae_decode/reference.py" (FastVideo): its module docstring
(sections "What is computed", "The first latent frame yields one frame",
"Causal caches", "Precision") and the interfaces of its functions.  It shares
no code with the CUDA path.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against brute force, closed forms, library routines or the pages' stated
invariants.  The composed network (``decode``) is pinned through its parts,
frame-loop = whole-sequence agreement, causality, batch independence and a
second, independently written whole-sequence composition from torch library
ops; there are no printed output values for it, so parity beyond composition
is unpinned.

``wan_tiled`` adds the tiled decode (the page "[Feature] Implement tiled VAE
encoding/decoding for Wan model. #11414"): per-tile ``decode`` plus seam
blending, pinned by ``tests/test_oracle_tiled.py``.  ``wan_latents`` adds the
latent de-normalisation in front of the decode, pinned by
``tests/test_oracle_latents.py``.
"""

from .wan_decode import (  # noqa: F401
    CACHE_T,
    PATCH_SIZE,
    attention,
    causal_conv,
    conv2d,
    decode,
    decode_chunk,
    decode_whole,
    dup_up,
    nearest_exact_up2,
    psnr,
    residual_block,
    rms_norm,
    round_bf16,
    silu,
    spatial_upsample,
    time_interleave,
    time_upsample,
    is_wan21,
    unpatchify,
)
from .wan_tiled import blend_tiles, decode_tiled, tile_origins  # noqa: F401
from .wan_latents import decode_normalized, denormalize_latents  # noqa: F401
