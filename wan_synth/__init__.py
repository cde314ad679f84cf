"""Seeded synthetic inputs for the Wan2.2-TI2V-5B VAE decode (and the Wan2.1
VAE decode, variant "wan21").

This module is shared by the CPU oracle and by the CUDA path's tests and
benchmark.  It holds no arithmetic of the decode itself: it only names the
decoder's parameters, gives their shapes, and draws seeded random values for
them and for the latents.

Parameter names and shapes follow the decoder description on the page
"wan22_vae_decode/reference.py" (FastVideo), module docstring section
"What is computed" and the functions ``decode_chunk``, ``up_block``,
``residual_block`` and ``attention``: conv weights are
[Cout, Cin, kt, kh, kw] (conv3d) or [Cout, Cin, kh, kw] (conv2d), biases are
[Cout], RMS-norm gammas are per-channel vectors of C values.

Random initialisation (the pages give none; this is the benchmark recipe):
conv weights and biases ~ U(-1/sqrt(fan_in), 1/sqrt(fan_in)) with
fan_in = Cin*kt*kh*kw of the conv, gammas = 1 + 0.1*N(0, 1), latents ~ N(0, 1).
Values are drawn with ``numpy.random.default_rng(seed)`` (PCG64), tensor by
tensor in the order of ``weight_names``; the generator is deterministic across
machines.

Variant "wan21" (the Wan2.1 VAE, z_dim 16): the pages give only its latent
channels and its 8x spatial compression; its other dimensions follow that
model's published configuration (base dim 96, up blocks 4b -> 4b, 2b -> 4b,
2b -> 2b, b -> b, resamplers halving the channels, conv_out to 3 colours),
with diffusers' parameter names (``upsamplers.0.*``).
"""

from __future__ import annotations

import functools

import numpy as np

Z_DIM = 48          # latent channels of the TI2V-5B VAE
OUT_PATCH_CH = 12   # conv_out channels: 3 colours x 2 x 2 patch
Z_DIM_WAN21 = 16    # latent channels of the Wan2.1 VAE
VARIANTS = ("ti2v", "wan21")

# (in-channel multiple, out-channel multiple, temporal upsampling, spatial
# upsampling) of the four up blocks, in units of the decoder base dim.
_UP = ((4, 4, True, True), (4, 4, True, True), (4, 2, False, True), (2, 1, False, False))
_RESNETS_PER_UP_BLOCK = 3


_UP_WAN21 = ((4, 4, True, True), (2, 4, True, True), (2, 2, False, True), (1, 1, False, False))


def up_blocks(base: int, variant: str = "ti2v"):
    """The four up blocks as (cin, cout, temporal, spatial) for a base dim."""
    table = _UP_WAN21 if variant == "wan21" else _UP
    return tuple((ci * base, co * base, t, s) for ci, co, t, s in table)


def weight_shapes(base: int = 256, variant: str = "ti2v") -> "dict[str, tuple[int, ...]]":
    """Ordered map name -> shape of the 110 decoder + post_quant_conv tensors
    (TI2V-5B), or of the Wan2.1 decoder's tensors (variant "wan21")."""
    if variant not in VARIANTS:
        raise ValueError(f"variant {variant!r}")
    wan21 = variant == "wan21"
    zd = Z_DIM_WAN21 if wan21 else Z_DIM
    c4 = 4 * base
    shapes: dict[str, tuple[int, ...]] = {}

    def conv3(name, co, ci, kt, kh, kw):
        shapes[f"{name}.weight"] = (co, ci, kt, kh, kw)
        shapes[f"{name}.bias"] = (co,)

    def conv2(name, co, ci, kh, kw):
        shapes[f"{name}.weight"] = (co, ci, kh, kw)
        shapes[f"{name}.bias"] = (co,)

    def resnet(name, ci, co):
        shapes[f"{name}.norm1.gamma"] = (ci,)
        conv3(f"{name}.conv1", co, ci, 3, 3, 3)
        shapes[f"{name}.norm2.gamma"] = (co,)
        conv3(f"{name}.conv2", co, co, 3, 3, 3)
        if ci != co:
            conv3(f"{name}.conv_shortcut", co, ci, 1, 1, 1)

    conv3("post_quant_conv", zd, zd, 1, 1, 1)
    conv3("decoder.conv_in", c4, zd, 3, 3, 3)
    resnet("decoder.mid_block.resnets.0", c4, c4)
    att = "decoder.mid_block.attentions.0"
    shapes[f"{att}.norm.gamma"] = (c4,)
    conv2(f"{att}.to_qkv", 3 * c4, c4, 1, 1)
    conv2(f"{att}.proj", c4, c4, 1, 1)
    resnet("decoder.mid_block.resnets.1", c4, c4)
    for i, (ci, co, temporal, spatial) in enumerate(up_blocks(base, variant)):
        name = f"decoder.up_blocks.{i}"
        ups = f"{name}.upsamplers.0" if wan21 else f"{name}.upsampler"
        c = ci
        for j in range(_RESNETS_PER_UP_BLOCK):
            resnet(f"{name}.resnets.{j}", c, co)
            c = co
        if temporal:
            conv3(f"{ups}.time_conv", 2 * co, co, 3, 1, 1)
        if spatial:
            conv2(f"{ups}.resample.1", co // 2 if wan21 else co, co, 3, 3)
    shapes["decoder.norm_out.gamma"] = (base,)
    conv3("decoder.conv_out", 3 if wan21 else OUT_PATCH_CH, base, 3, 3, 3)
    return shapes


def weight_names(base: int = 256, variant: str = "ti2v") -> "list[str]":
    return list(weight_shapes(base, variant))


def _fan_in(shape) -> int:
    return int(np.prod(shape[1:]))


@functools.lru_cache(maxsize=4)
def _weights_cached(base: int, seed: int, variant: str):
    rng = np.random.default_rng(seed)
    shapes = weight_shapes(base, variant)
    out: dict[str, np.ndarray] = {}
    for name, shape in shapes.items():
        n = int(np.prod(shape))
        if name.endswith(".gamma"):
            g = rng.standard_normal(n, dtype=np.float32)
            out[name] = (np.float32(1.0) + np.float32(0.1) * g).reshape(shape)
            continue
        wshape = shapes[name.rsplit(".", 1)[0] + ".weight"]
        bound = np.float32(1.0 / np.sqrt(_fan_in(wshape)))
        # drawn flat, then shaped (numpy is much slower on n-d shapes)
        u = rng.random(n, dtype=np.float32).reshape(shape)
        u *= np.float32(2.0)
        u -= np.float32(1.0)
        u *= bound
        out[name] = u
    for v in out.values():
        v.setflags(write=False)
    return out


def make_weights(base: int = 256, seed: int = 0, variant: str = "ti2v") -> "dict[str, np.ndarray]":
    """Seeded random-init weight table (fp32 numpy arrays, read-only)."""
    return dict(_weights_cached(base, seed, variant))


def make_latents(shape, seed: int) -> np.ndarray:
    """Latents [B, 48, T, h, w] ~ N(0, 1), fp32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(tuple(shape))


def make_normal(shape, seed: int) -> np.ndarray:
    """Any tensor ~ N(0, 1), fp32 (e.g. the attention block's input)."""
    return make_latents(shape, seed)


# The workloads of the benchmark and the parity tests (synthetic, seeded).
CONFIGS = {
    # tiny-width decoder, for the oracle in seconds
    "tiny": dict(base=16, latents=(1, 48, 2, 4, 4), weight_seed=0, latent_seed=1),
    # full-width decoder at a small resolution
    "small": dict(base=256, latents=(1, 48, 3, 16, 16), weight_seed=0, latent_seed=1),
    # isolated mid-block attention: x [frames, C, h, w]
    "attention": dict(base=256, x=(8, 1024, 44, 80), weight_seed=0, x_seed=2),
    # 704x1280, 121 frames
    "720p": dict(base=256, latents=(1, 48, 31, 44, 80), weight_seed=0, latent_seed=3),
    # 1280x704 portrait, 81 frames
    "portrait": dict(base=256, latents=(1, 48, 21, 80, 44), weight_seed=0, latent_seed=4),
    # 480x832, batch 2, 81 frames
    "480p_b2": dict(base=256, latents=(2, 48, 21, 30, 52), weight_seed=0, latent_seed=5),
    # the Wan2.1 VAE (z_dim 16, 8x spatial): tiny width, full width small, 720p
    "wan21_tiny": dict(base=16, variant="wan21", latents=(1, 16, 2, 4, 4), weight_seed=0, latent_seed=1),
    "wan21_small": dict(base=96, variant="wan21", latents=(1, 16, 3, 16, 16), weight_seed=0, latent_seed=1),
    "wan21_720p": dict(base=96, variant="wan21", latents=(1, 16, 21, 90, 160), weight_seed=0, latent_seed=6),
}
