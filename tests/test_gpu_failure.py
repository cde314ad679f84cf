"""Failure detection on the GPU without a fault: a conv kernel whose producer
withholds one stage runs out its (shortened) bounded wait, drains and exits;
the library reports WAN_ERR_INTERNAL with the device error code, and the
context keeps working (a normal conv afterwards is checked against the
oracle).  Covered: the implicit-GEMM conv kernel in its one-CTA, cluster-pair
and row-tile forms, conv_out's tap-folded kernel, and both flash attention
kernels (one CTA per 128 queries; C / 256 CTAs per 128 queries)."""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import lib_ready, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cout", [64, 256, 96, 12], ids=["one_cta", "cluster_of_two", "row_tiles_pair", "conv_out"])
def test_bounded_wait_expires_and_is_reported(cout):
    wv = lib_ready()
    lib = wv.load()
    code = ctypes.c_int32(0)
    status = lib.wan_selftest_wait_timeout(cout, ctypes.byref(code), None)
    assert status == 9, (status, lib.wan_vae_last_error())        # WAN_ERR_INTERNAL
    assert code.value in (1, 2, 3)
    assert b"bounded wait" in lib.wan_vae_last_error()
    # the context is still usable: the same kernel run normally right after is correct
    rng = np.random.default_rng(5)
    x = oracle.round_bf16(rng.standard_normal((1, 3, 8, 16, 64)))
    w = oracle.round_bf16(rng.uniform(-1, 1, (cout, 64, 3, 3, 3)) / math.sqrt(64 * 27))
    b = oracle.round_bf16(rng.uniform(-0.1, 0.1, cout))
    xn = x.transpose(0, 4, 1, 2, 3)
    ref = oracle.causal_conv(xn[:, :, 2:], w, b, xn[:, :, :2])
    if cout == 12:
        _, got = wv.conv_out_video(to_dev(x, torch.bfloat16), 2, to_dev(w), to_dev(b), preclamp=True)
        got, ref = got.cpu().numpy(), oracle.unpatchify(ref)
        assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
    else:
        got = wv.causal_conv3d(to_dev(x, torch.bfloat16), 2, to_dev(w), to_dev(b)).float().cpu().numpy()
        ref = ref.transpose(0, 2, 3, 4, 1)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max())


@pytest.mark.parametrize("C", [384, 1024], ids=["flash_one_cta", "flash_four_ctas"])
def test_flash_attention_bounded_wait_expires_and_is_reported(C):
    wv = lib_ready()
    lib = wv.load()
    code = ctypes.c_int32(0)
    status = lib.wan_selftest_attention_timeout(C, ctypes.byref(code), None)
    assert status == 9, (status, lib.wan_vae_last_error())        # WAN_ERR_INTERNAL
    assert code.value in (1, 2, 3)
    assert b"bounded wait" in lib.wan_vae_last_error()
    # the context is still usable: the attention block at the same width is right
    from tests.test_gpu_kernels import _attention_check
    _attention_check(wv, N=1, C=C, H=9, W=23, frames=[0], seed=19)
