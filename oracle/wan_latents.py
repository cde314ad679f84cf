"""Latent de-normalisation in front of the decode (CPU oracle; test
infrastructure only, the CUDA path never imports it).

Source: the page "[Feature] Implement tiled VAE encoding/decoding for Wan
model. #11414" (diffusers pull request), where the Wan VAE keeps two
per-channel lists in its configuration, ``latents_mean`` and
``latents_std``, used by downstream code to map between the VAE's latent
scale and the standardised latents a diffusion model works in.  The page
shows that they exist (one value per latent channel) but not their values or
the formula.  Reading taken: latents are standardised per channel as
(x - mean) / std, so de-normalisation, the step in front of the decode, is
its inverse x = z * std + mean, per latent channel c, broadcast over batch,
frames and positions.  For a bf16 decode the de-normalised latents are what
the bf16 contract rounds.
"""

from __future__ import annotations

import numpy as np

from .wan_decode import decode


def denormalize_latents(z, mean, std) -> np.ndarray:
    """z [B, C, T, h, w] -> z * std[c] + mean[c], computed in fp64, returned fp32."""
    z = np.asarray(z, np.float64)
    C = z.shape[1]
    mean = np.asarray(mean, np.float64).reshape(-1)
    std = np.asarray(std, np.float64).reshape(-1)
    if mean.shape != (C,) or std.shape != (C,):
        raise ValueError(f"need {C} means and {C} stds, got {mean.shape} and {std.shape}")
    shape = (1, C) + (1,) * (z.ndim - 2)
    return (z * std.reshape(shape) + mean.reshape(shape)).astype(np.float32)


def decode_normalized(z, weights, mean, std, chunk: int = 1, round_latents=None) -> np.ndarray:
    """``decode`` of the de-normalised latents.  ``round_latents``, if given,
    is applied to them first (the bf16 contract's rounding)."""
    x = denormalize_latents(z, mean, std)
    if round_latents is not None:
        x = round_latents(x)
    return decode(x, weights, chunk=chunk)
