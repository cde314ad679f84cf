"""Layer parity on the GPU: the tensor-core causal conv and the attention
block, through the C ABI, against the CPU oracle on the same bf16 inputs."""

import math

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import lib_ready, to_dev
from tests.parity_log import record

pytestmark = pytest.mark.gpu
RNG = np.random.default_rng(77)


@pytest.fixture(scope="module")
def wv():
    return lib_ready()


def _bf(a):
    return oracle.round_bf16(np.asarray(a, np.float32))


# (B, n_hist, F, H, W, Cin, Cout, kernel): tiles of 16x8 positions, ragged
# edges, channel counts off the 64-block, 1/2 history frames, all kernel shapes
CONV_CASES = [
    (1, 0, 1, 8, 16, 64, 64, (3, 3, 3)),
    (1, 2, 2, 12, 20, 48, 256, (3, 3, 3)),
    (2, 1, 2, 30, 52, 128, 128, (3, 3, 3)),
    (1, 2, 3, 9, 17, 256, 512, (3, 1, 1)),
    (1, 0, 2, 5, 7, 64, 16, (1, 1, 1)),
    (1, 2, 2, 17, 33, 256, 16, (3, 3, 3)),
    (1, 0, 1, 11, 24, 1024, 256, (3, 3, 3)),
    (1, 1, 1, 4, 4, 16, 32, (3, 3, 3)),
    (1, 0, 2, 19, 21, 512, 512, (1, 3, 3)),
    # the Wan2.1 widths: N tiles of 96 and 192, K padded from 96 to 128
    (1, 2, 2, 13, 22, 96, 96, (3, 3, 3)),
    (1, 1, 2, 10, 18, 192, 192, (3, 3, 3)),
    (2, 0, 1, 9, 14, 192, 384, (3, 3, 3)),
]


@pytest.mark.parametrize("case", CONV_CASES, ids=lambda c: "B{}h{}F{}_{}x{}_{}to{}_k{}{}{}".format(*c[:7], *c[7]))
def test_causal_conv_vs_oracle(wv, case):
    B, nh, F, H, W, Cin, Cout, k = case
    x = _bf(RNG.standard_normal((B, nh + F, H, W, Cin)))
    w = _bf(RNG.uniform(-1, 1, (Cout, Cin, *k)) / math.sqrt(Cin * np.prod(k)))
    b = _bf(RNG.uniform(-0.1, 0.1, Cout))
    got = wv.causal_conv3d(to_dev(x, torch.bfloat16), nh, to_dev(w), to_dev(b)).float().cpu().numpy()
    torch.cuda.synchronize()
    xn = x.transpose(0, 4, 1, 2, 3)                      # NCDHW
    ref = oracle.causal_conv(xn[:, :, nh:], w, b, xn[:, :, :nh] if nh else None).transpose(0, 2, 3, 4, 1)
    # fp32 accumulation of exact bf16 products; the output is rounded to bf16
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()), float(err.max())


def _attn_weights(C, seed, qkv_scale=1.0):
    r = np.random.default_rng(seed)
    return {
        "a.norm.gamma": _bf(1 + 0.1 * r.standard_normal(C)),
        "a.to_qkv.weight": _bf(qkv_scale * r.uniform(-1, 1, (3 * C, C, 1, 1)) / math.sqrt(C)),
        "a.to_qkv.bias": _bf(r.uniform(-1, 1, 3 * C) / math.sqrt(C)),
        "a.proj.weight": _bf(r.uniform(-1, 1, (C, C, 1, 1)) / math.sqrt(C)),
        "a.proj.bias": _bf(r.uniform(-1, 1, C) / math.sqrt(C)),
    }


def _attention_check(wv, N, C, H, W, frames, seed, qkv_scale=1.0, rel_tol=1e-2, abs_tol=4e-2):
    w = _attn_weights(C, seed, qkv_scale)
    x = _bf(np.random.default_rng(seed + 1).standard_normal((N, H * W, C)))
    got = wv.attention_block(to_dev(x, torch.bfloat16), {k: to_dev(v) for k, v in w.items()}, H, W)
    got = got.float().cpu().numpy()
    for f in frames:
        xf = x[f].reshape(H, W, C).transpose(2, 0, 1)[None, :, None]    # [1, C, 1, H, W]
        ref = oracle.attention(xf, w, "a")[0, :, 0].transpose(1, 2, 0).reshape(H * W, C)
        err = np.abs(got[f] - ref)
        rel = np.linalg.norm(got[f] - ref) / np.linalg.norm(ref)
        record(f"attention block C={C} {H}x{W} frame {f} (bf16)", float(err.max()), None, rel_l2=float(rel))
        assert err.max() <= abs_tol and rel <= rel_tol, (f, float(err.max()), float(rel))


def test_attention_small(wv):
    _attention_check(wv, N=3, C=64, H=4, W=9, frames=range(3), seed=5)


def test_attention_ragged_positions(wv):
    _attention_check(wv, N=2, C=128, H=7, W=23, frames=range(2), seed=6)


# Head dims up to 384 run the flash kernel (scores never leave the SM): key
# blocks of 128 with a ragged last one, V^T row groups of 128 (C = 384) and of
# 64 (C = 192, 320), a frame of fewer than 128 positions.
@pytest.mark.parametrize("N,C,H,W", [(2, 384, 13, 29), (1, 192, 10, 26), (1, 320, 9, 15), (3, 384, 5, 7)],
                         ids=lambda v: str(v))
def test_attention_flash_widths(wv, N, C, H, W):
    _attention_check(wv, N=N, C=C, H=H, W=W, frames=range(N), seed=11)


def test_attention_flash_large_logits(wv):
    """qkv weights 4x larger (logits 16x): over 4800 keys the row maxima of
    later key blocks exceed the first block's by more than the rescale
    threshold (8 in log2 units) for many rows, so the running max moves and
    the output accumulator is rescaled.  The GPU stores q and k in bf16 (the
    oracle keeps them in fp32): a rounding of 2^-9 relative moves a logit of
    30 by about 0.06, and the sharper softmax passes that on to the output,
    so the bounds here are max |diff| <= 0.15 and relative L2 <= 2e-2 (a
    wrong rescale factor would put whole rows off by O(1))."""
    _attention_check(wv, N=1, C=384, H=60, W=80, frames=[0], seed=12, qkv_scale=4.0, rel_tol=2e-2, abs_tol=0.15)


# Head dims 512 and 1024 run the four-CTA flash kernel (C / 256 CTAs per 128
# queries, each with 256 output columns; key blocks of 256): ragged last key
# and query blocks, exactly one key block, frames of fewer than 128 positions,
# and frames of one position (one key: the output is proj(v) + x).
@pytest.mark.parametrize("N,C,H,W", [(2, 1024, 13, 29), (1, 512, 10, 26), (3, 1024, 5, 7), (1, 512, 16, 16),
                                     (1, 1024, 9, 57), (2, 1024, 1, 1), (1, 512, 1, 1)], ids=lambda v: str(v))
def test_attention_flash_split_widths(wv, N, C, H, W):
    _attention_check(wv, N=N, C=C, H=H, W=W, frames=range(N), seed=16)


def test_attention_flash_split_large_logits(wv):
    """As the large-logit case above, at head dim 1024 (the cluster kernel):
    1200 keys in 5 blocks of 256, qkv weights 4x larger, so the running max
    moves and each CTA rescales its output columns; same bounds and reason."""
    _attention_check(wv, N=1, C=1024, H=30, W=40, frames=[0], seed=17, qkv_scale=4.0, rel_tol=2e-2, abs_tol=0.15)


def test_attention_gemm_path_width(wv):
    """A head dim no flash kernel takes (768) runs the score GEMM, row
    softmax and P V GEMM path."""
    _attention_check(wv, N=2, C=768, H=11, W=27, frames=range(2), seed=18)


def test_attention_flash_wan21_720p_frame(wv):
    """Wan2.1's mid block at 720p: 90 x 160 = 14,400 positions, C = 384, one
    frame against the oracle (113 key blocks)."""
    _attention_check(wv, N=1, C=384, H=90, W=160, frames=[0], seed=13)


def test_attention_handle_matches_one_shot(wv):
    """Weights packed once (wan_attention_create) and run twice give the
    one-shot entry point's result bit for bit, for each path (flash at C =
    384, the cluster flash kernel at C = 1024, score GEMMs at C = 768)."""
    for N, C, H, W in ((2, 384, 12, 20), (1, 1024, 8, 12), (1, 768, 8, 12)):
        w = {k: to_dev(v) for k, v in _attn_weights(C, 14).items()}
        x = to_dev(_bf(np.random.default_rng(15).standard_normal((N, H * W, C))), torch.bfloat16)
        ref = wv.attention_block(x, w, H, W)
        blk = wv.AttentionBlock(w, N, H, W, C)
        for _ in range(2):
            got = blk(x)
            blk.sync_status()
            assert torch.equal(got, ref), C
        blk.close()


def test_attention_full_width_720p_frames(wv):
    """The isolated attention block at its full size: 8 frames of 44x80
    positions, C = 1024; frames 0 and 7 checked against the oracle."""
    _attention_check(wv, N=8, C=1024, H=44, W=80, frames=(0, 7), seed=2)


# conv_out as the bf16 decode runs it (spatial taps folded into N, 16 x 16
# input boxes with 14 x 14 outputs each): (B, n_hist, F, H, W, Cin, Cout).
# 256 -> 12 with the 2 x 2 unpatchify (TI2V-5B) and 96 -> 3 (Wan2.1, a 64-channel
# block holding 32); ragged boxes at both edges, history 0/1/2, a frame
# smaller than one box, exactly one box, and 16 input channels (one block of
# which 48 channels are TMA zero fill).
VIDEO_CASES = [
    (1, 2, 2, 17, 33, 256, 12),
    (2, 0, 1, 30, 29, 256, 12),
    (1, 1, 3, 8, 16, 256, 12),
    (1, 2, 2, 1, 5, 256, 12),
    (1, 2, 2, 45, 20, 96, 3),
    (1, 0, 1, 14, 14, 16, 12),
]


@pytest.mark.parametrize("case", VIDEO_CASES, ids=lambda c: "B{}h{}F{}_{}x{}_{}to{}".format(*c))
def test_conv_out_video_vs_oracle(wv, case):
    B, nh, F, H, W, Cin, Cout = case
    x = _bf(RNG.standard_normal((B, nh + F, H, W, Cin)))
    w = _bf(RNG.uniform(-1, 1, (Cout, Cin, 3, 3, 3)) / math.sqrt(Cin * 27) * 4.0)
    b = _bf(RNG.uniform(-0.1, 0.1, Cout))
    got, pre = wv.conv_out_video(to_dev(x, torch.bfloat16), nh, to_dev(w), to_dev(b), preclamp=True)
    torch.cuda.synchronize()
    got, pre = got.float().cpu().numpy(), pre.cpu().numpy()
    xn = x.transpose(0, 4, 1, 2, 3)                      # NCDHW
    conv = oracle.causal_conv(xn[:, :, nh:], w, b, xn[:, :, :nh] if nh else None)
    ref_pre = oracle.unpatchify(conv) if Cout == 12 else conv
    ref = np.clip(ref_pre, -1.0, 1.0)
    assert pre.shape == ref_pre.shape and got.shape == ref.shape
    # fp32 accumulation of exact bf16 products, in another order than the oracle's
    err_pre = np.abs(pre - ref_pre)
    assert err_pre.max() <= 1e-4 * np.abs(ref_pre).max(), float(err_pre.max())
    # the clamped video is rounded to bf16
    err = np.abs(got - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6), float(err.max())
    record(f"conv_out video {H}x{W} {Cin}->{Cout} (bf16 in)", float(err.max()), None,
           preclamp_max_abs=float(err_pre.max()))
