"""Whole-decode parity on the GPU through the C ABI against the CPU oracle.

The bf16 decode is fed the same latents and weights; the oracle receives
them rounded to bf16 (the first step of the bf16 contract) and computes in
fp32.  Bar: max |diff| <= 4e-2 and PSNR >= 40 dB on the clamped video.
"""

import numpy as np
import pytest
import torch

import oracle
import wan_synth
from tests.gpu_util import lib_ready, rounded, to_dev, weights_dev
from tests.parity_log import record

pytestmark = pytest.mark.gpu
TOL, PSNR_MIN = 4e-2, 40.0
TOL_F32 = 2e-3


@pytest.fixture(scope="module")
def wv():
    return lib_ready()


@pytest.fixture(scope="module")
def tiny():
    w = wan_synth.make_weights(base=16, seed=0)
    return w, weights_dev(w)


@pytest.fixture(scope="module")
def small():
    w = wan_synth.make_weights(base=256, seed=0)
    return w, weights_dev(w)


def _ref(z, w):
    return oracle.decode(oracle.round_bf16(z), rounded(w))


def _check(got, ref, case=None):
    err = float(np.abs(got - ref).max())
    p = oracle.psnr(got, ref)
    if case:
        record(case, err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)
    return err, p


def _decode(wv, model, z, chunk, out_dtype=torch.float32):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    v = st.decode_clip(to_dev(z), out_dtype=out_dtype)
    st.sync_status()
    return v.float().cpu().numpy()


@pytest.mark.parametrize("chunk", [1, 2])
def test_tiny_decode(wv, tiny, chunk):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=1)
    model = wv.Model(wd, dtype=torch.bfloat16)
    _check(_decode(wv, model, z, chunk), _ref(z, w), f"tiny [1,48,2,4,4] bf16 chunk {chunk}")


def test_tiny_ragged_batch_and_first_chunk_rules(wv, tiny):
    """B = 2, a non-square latent, T = 3 decoded in chunks of 2: the first
    chunk holds two latent frames (time conv on its second frame only)."""
    w, wd = tiny
    z = wan_synth.make_latents((2, 48, 3, 5, 6), seed=3)
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = _decode(wv, model, z, 2)
    assert got.shape == (2, 3, 9, 80, 96)
    _check(got, _ref(z, w), "tiny [2,48,3,5,6] bf16 chunk 2")
    # batch independence: each sample alone gives the same frames bit for bit
    one = _decode(wv, model, z[1:2], 2)
    np.testing.assert_array_equal(one, got[1:2])


def test_tiny_chunk_api_and_preclamp(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 3, 4, 4), seed=4)
    model = wv.Model(wd, dtype=torch.bfloat16)
    st = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    out = torch.zeros((1, 3, 9, 64, 64), device="cuda")
    pre = torch.zeros_like(out)
    zt = to_dev(z)
    st.reset()
    st.decode_chunk(zt, 0, 1, out, 0, preclamp=pre)     # 1 frame
    st.decode_chunk(zt, 1, 2, out, 1, preclamp=pre)     # 8 frames
    st.sync_status()
    ref_clamped, ref_pre = oracle.decode(oracle.round_bf16(z), rounded(w), return_preclamp=True)
    _check(out.cpu().numpy(), ref_clamped)
    assert float(np.abs(pre.cpu().numpy() - ref_pre).max()) <= TOL
    assert float(out.abs().max()) <= 1.0


def test_tiny_one_shot_and_host_paths(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=1)
    v1 = wv.decode(to_dev(z), wd, dtype=torch.bfloat16).float().cpu().numpy()
    _check(v1, _ref(z, w))
    model = wv.Model(wd, dtype=torch.bfloat16)
    st = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    dev = st.decode_clip(to_dev(z), out_dtype=torch.bfloat16)
    host = torch.empty((1, 3, 5, 64, 64), dtype=torch.bfloat16).pin_memory()
    st.decode_clip_host(torch.from_numpy(z).pin_memory(), host)
    torch.cuda.synchronize()
    assert torch.equal(host, dev.cpu())          # same kernels, same chunking: bit-exact
    # second call on the same stream: reused staging, three chunks (both
    # buffers recycled), another clip length and fp32 output
    z5 = wan_synth.make_latents((1, 48, 5, 4, 4), seed=2)
    dev5 = st.decode_clip(to_dev(z5), out_dtype=torch.float32)
    host5 = torch.empty((1, 3, 17, 64, 64), dtype=torch.float32).pin_memory()
    st.decode_clip_host(torch.from_numpy(z5).pin_memory(), host5)
    torch.cuda.synchronize()
    assert torch.equal(host5, dev5.cpu())


def test_determinism(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=2)
    model = wv.Model(wd, dtype=torch.bfloat16)
    a = _decode(wv, model, z, 2)
    b = _decode(wv, model, z, 2)
    np.testing.assert_array_equal(a, b)


@pytest.fixture(scope="module")
def small_ref(small):
    w, _ = small
    z = wan_synth.make_latents((1, 48, 3, 16, 16), seed=1)
    return z, _ref(z, w)


@pytest.mark.parametrize("chunk", [1, 3])
def test_full_width_small_decode(wv, small, small_ref, chunk):
    """Full-width TI2V-5B decoder (channels 1024/1024/512/256), latents
    [1, 48, 3, 16, 16] -> video [1, 3, 9, 256, 256]."""
    _, wd = small
    z, ref = small_ref
    model = wv.Model(wd, dtype=torch.bfloat16)
    _check(_decode(wv, model, z, chunk), ref, f"full-width [1,48,3,16,16] bf16 chunk {chunk}")


# ------------------------------------------------------------------ fp32
def _check_f32(got, pre, ref_clamped, ref_pre, case=None):
    e1 = float(np.abs(got - ref_clamped).max())
    e2 = float(np.abs(pre - ref_pre).max())
    if case:
        record(case, e1, oracle.psnr(got, ref_clamped), preclamp_max_abs=e2)
    assert e1 <= TOL_F32 and e2 <= TOL_F32, (e1, e2)
    return e1, e2


def _decode_f32(wv, model, z, chunk):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    pre = torch.empty((B, 3, 4 * T - 3, 16 * h, 16 * w), device="cuda")
    v = st.decode_clip(to_dev(z), out_dtype=torch.float32, preclamp=pre)
    st.sync_status()
    return v.cpu().numpy(), pre.cpu().numpy()


@pytest.mark.parametrize("chunk", [1, 2])
def test_tiny_decode_fp32(wv, tiny, chunk):
    """fp32 decode (bf16 hi/lo pairs on the tensor cores) against the fp32
    oracle on the unrounded inputs: within 2e-3 before and after the clamp."""
    w, wd = tiny
    z = wan_synth.make_latents((2, 48, 3, 4, 5), seed=11)
    model = wv.Model(wd, dtype=torch.float32)
    got, pre = _decode_f32(wv, model, z, chunk)
    ref, ref_pre = oracle.decode(z, w, return_preclamp=True)
    _check_f32(got, pre, ref, ref_pre, f"tiny [2,48,3,4,5] fp32 chunk {chunk}")


def test_full_width_small_decode_fp32(wv, small):
    w, wd = small
    z = wan_synth.make_latents((1, 48, 3, 16, 16), seed=1)
    model = wv.Model(wd, dtype=torch.float32)
    got, pre = _decode_f32(wv, model, z, 2)
    ref, ref_pre = oracle.decode(z, w, return_preclamp=True)
    _check_f32(got, pre, ref, ref_pre, "full-width [1,48,3,16,16] fp32 chunk 2")


# ------------------------------------------------------------- edge cases
def test_single_latent_frame(wv, tiny):
    """T = 1: one output frame, no time conv ever runs (first-chunk rule)."""
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 1, 4, 4), seed=21)
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = _decode(wv, model, z, 4)
    assert got.shape == (1, 3, 1, 64, 64)
    _check(got, _ref(z, w), "tiny T=1 bf16")


@pytest.mark.parametrize("h,w", [(1, 1), (2, 3), (1, 5)])
def test_frames_with_few_positions(wv, tiny, h, w):
    """Latent frames of fewer than 16 positions (down to one): the attention's
    score GEMM then covers more key rows than the frame has."""
    wt, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, h, w), seed=22)
    for dt in (torch.bfloat16, torch.float32):
        model = wv.Model(wd, dtype=dt)
        got = _decode(wv, model, z, 2)
        assert got.shape == (1, 3, 5, 16 * h, 16 * w)
        if dt == torch.bfloat16:
            _check(got, _ref(z, wt), f"tiny {h}x{w} latents bf16")
        else:
            err = float(np.abs(got - oracle.decode(z, wt)).max())
            record(f"tiny {h}x{w} latents fp32", err, None)
            assert err <= TOL_F32, err


def test_stream_reuse_after_reset(wv, tiny):
    """A stream decodes a second clip from scratch: bit-identical to a fresh stream."""
    w, wd = tiny
    za = wan_synth.make_latents((1, 48, 3, 4, 4), seed=22)
    zb = wan_synth.make_latents((1, 48, 3, 4, 4), seed=23)
    model = wv.Model(wd, dtype=torch.bfloat16)
    st = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    st.decode_clip(to_dev(za), out_dtype=torch.float32)
    second = st.decode_clip(to_dev(zb), out_dtype=torch.float32).cpu().numpy()
    st.sync_status()
    np.testing.assert_array_equal(second, _decode(wv, model, zb, 2))


def test_chunk_argument_errors(wv, tiny):
    _, wd = tiny
    model = wv.Model(wd, dtype=torch.bfloat16)
    st = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    z = to_dev(wan_synth.make_latents((1, 48, 3, 4, 4), seed=24))
    out = torch.zeros((1, 3, 9, 64, 64), device="cuda")
    st.reset()
    with pytest.raises(wv.WanError) as e:
        st.decode_chunk(z, 0, 3, out, 0)            # more frames than max_chunk
    assert e.value.status == 1
    with pytest.raises(wv.WanError):
        st.decode_chunk(z, 2, 2, out, 0)            # frames past the end of z
    with pytest.raises(wv.WanError):
        st.decode_chunk(z, 0, 2, out, 8)            # output frames past the end of out
    st.decode_chunk(z, 0, 2, out, 0)                # valid calls still work afterwards
    st.sync_status()


def test_one_shot_fp32(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 48, 2, 4, 4), seed=25)
    got = wv.decode(to_dev(z), wd, dtype=torch.float32).cpu().numpy()
    ref = oracle.decode(z, w)
    assert float(np.abs(got - ref).max()) <= TOL_F32


def test_checkpoint_resume(wv, tiny):
    """Save the stream's state after the first chunk, resume in a fresh stream:
    the resumed frames equal the uninterrupted decode bit for bit."""
    _, wd = tiny
    z = to_dev(wan_synth.make_latents((1, 48, 4, 4, 4), seed=26))
    model = wv.Model(wd, dtype=torch.bfloat16)
    a = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    full = torch.zeros((1, 3, 13, 64, 64), device="cuda")
    a.reset()
    a.decode_chunk(z, 0, 2, full, 0)            # frames 0..4
    state = a.save_state()
    a.decode_chunk(z, 2, 2, full, 5)            # frames 5..12
    b = wv.DecodeStream(model, 1, 4, 4, max_chunk=2)
    b.load_state(state)
    resumed = torch.zeros_like(full)
    b.decode_chunk(z, 2, 2, resumed, 5)
    a.sync_status()
    b.sync_status()
    assert torch.equal(resumed[:, :, 5:], full[:, :, 5:])
    # a state does not load into a stream of another shape
    c = wv.DecodeStream(model, 1, 4, 5, max_chunk=2)
    with pytest.raises(wv.WanError):
        c.load_state(state)
