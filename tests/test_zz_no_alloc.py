"""The allocation-free causal conv (wan_causal_conv3d_noalloc) against the
allocating one (wan_causal_conv3d), through the C ABI.

It serves callers that may not allocate device memory themselves (a host
framework owning every byte of GPU memory through its own pool, or a
latency-critical path that cannot afford cudaMalloc's implicit device
synchronisation); its scratch is a fixed array inside the library, shared by
every call.  Two calls in a row with different shapes check that the second
call does not see the first call's leftovers (history slots, channel
padding).  This file is collected last on purpose.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import lib_ready, to_dev

pytestmark = pytest.mark.gpu


def _bf(a):
    return oracle.round_bf16(np.asarray(a, np.float32))


# (B, n_hist, F, H, W, Cin, Cout, kernel): the second call has fewer input
# channels (48, padded to 64) and no history, where the first had 64 and 2.
CALLS = [
    (1, 2, 2, 12, 20, 64, 128, (3, 3, 3)),
    (2, 0, 1, 9, 17, 48, 64, (3, 3, 3)),
]


def test_noalloc_conv_matches_allocating_conv_two_calls():
    wv = lib_ready()
    lib = wv.load()
    rng = np.random.default_rng(2024)
    stream = torch.cuda.current_stream()
    for B, nh, F, H, W, Cin, Cout, k in CALLS:
        x = to_dev(_bf(rng.standard_normal((B, nh + F, H, W, Cin))), torch.bfloat16)
        w = to_dev(_bf(rng.uniform(-1, 1, (Cout, Cin, *k)) / math.sqrt(Cin * np.prod(k))))
        b = to_dev(_bf(rng.uniform(-0.1, 0.1, Cout)))
        ref = wv.causal_conv3d(x, nh, w, b).float()
        out = torch.full((B, F, H, W, Cout), float("nan"), device="cuda", dtype=torch.bfloat16)
        status = lib.wan_causal_conv3d_noalloc(x.data_ptr(), B, nh, F, H, W, Cin, w.data_ptr(), b.data_ptr(), 0,
                                               Cout, *k, out.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert status == 0, lib.wan_vae_last_error()
        torch.cuda.synchronize()
        got = out.float()
        assert torch.isfinite(got).all()
        err = (got - ref).abs()
        tol = 2.0 ** -8 * ref.abs() + 1e-3 * ref.abs().max()
        assert bool((err <= tol).all()), float(err.max())


def test_noalloc_conv_rejects_oversize_scratch():
    wv = lib_ready()
    lib = wv.load()
    # 1024 -> 1024 3x3x3 needs 56 MiB of packed weights: over the 32 MiB limit;
    # rejected on the host before any work is enqueued (pointers unused)
    vp = ctypes.c_void_p
    status = lib.wan_causal_conv3d_noalloc(vp(16), 1, 0, 1, 8, 8, 1024, vp(16), vp(16), 0, 1024, 3, 3, 3, vp(16),
                                           None)
    assert status == 5
    assert b"scratch" in lib.wan_vae_last_error()
