"""The allocation-free causal conv (wan_causal_conv3d_noalloc) through the C
ABI, against the CPU oracle's causal conv and against the allocating entry
point (wan_causal_conv3d).

It serves callers that may not allocate device memory themselves (a host
framework owning every byte of GPU memory through its own pool, or a
latency-critical path that cannot afford cudaMalloc's implicit device
synchronisation); its scratch is a fixed array inside the library, shared by
every call.  Calls in a row with different shapes check that a call does not
see an earlier call's leftovers (history slots, channel padding, weight
padding); output widths of 80 and 320 channels leave the last N tile of the
kernel partly unused.  This file is collected last on purpose.
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


# (B, n_hist, F, H, W, Cin, Cout, kernel), run in this order: fewer input
# channels (48, padded to 64) and no history after 64 channels and two history
# frames; then output widths that are not whole N tiles (80 in a 128-wide
# tile, 320 = one 256-wide tile and a quarter of the next), a 3x1x1 time conv.
CALLS = [
    (1, 2, 2, 12, 20, 64, 128, (3, 3, 3)),
    (2, 0, 1, 9, 17, 48, 64, (3, 3, 3)),
    (1, 1, 2, 11, 19, 96, 80, (3, 3, 3)),
    (1, 2, 1, 10, 21, 64, 320, (3, 3, 3)),
    (1, 2, 2, 7, 9, 128, 320, (3, 1, 1)),
]


def _tol(ref):
    # fp32 accumulation of exact bf16 products; the output is rounded to bf16
    return 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()


def test_noalloc_conv_matches_oracle_and_allocating_conv():
    wv = lib_ready()
    lib = wv.load()
    rng = np.random.default_rng(2024)
    stream = torch.cuda.current_stream()
    for B, nh, F, H, W, Cin, Cout, k in CALLS:
        x = _bf(rng.standard_normal((B, nh + F, H, W, Cin)))
        w = _bf(rng.uniform(-1, 1, (Cout, Cin, *k)) / math.sqrt(Cin * np.prod(k)))
        b = _bf(rng.uniform(-0.1, 0.1, Cout))
        xd, wd, bd = to_dev(x, torch.bfloat16), to_dev(w), to_dev(b)
        out = torch.full((B, F, H, W, Cout), float("nan"), device="cuda", dtype=torch.bfloat16)
        status = lib.wan_causal_conv3d_noalloc(xd.data_ptr(), B, nh, F, H, W, Cin, wd.data_ptr(), bd.data_ptr(), 0,
                                               Cout, *k, out.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert status == 0, lib.wan_vae_last_error()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        # the oracle: causal conv in NCDHW with the first nh frames as history
        xn = x.transpose(0, 4, 1, 2, 3)
        ref = oracle.causal_conv(xn[:, :, nh:], w, b, xn[:, :, :nh] if nh else None).transpose(0, 2, 3, 4, 1)
        err = np.abs(got - ref)
        assert np.all(err <= _tol(ref)), (Cout, float(err.max()))
        # the allocating entry point on the same inputs
        alloc = wv.causal_conv3d(xd, nh, wd, bd).float().cpu().numpy()
        err = np.abs(got - alloc)
        assert np.all(err <= _tol(alloc)), (Cout, float(err.max()))


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
