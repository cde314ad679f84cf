"""Helpers of the GPU parity tests (marshalling between NumPy and torch)."""

import numpy as np
import torch

import oracle


def lib_ready():
    from video_vae_decoding_gb300 import build
    build.build()
    import video_vae_decoding_gb300 as wv
    wv.load()
    return wv


def to_dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dtype)


def weights_dev(w):
    return {k: to_dev(v) for k, v in w.items()}


def rounded(w):
    """The bf16 contract's inputs: every weight rounded to bf16 (as fp32)."""
    return {k: oracle.round_bf16(v) for k, v in w.items()}
