"""The Wan2.1 VAE decode (z_dim 16, 8x spatial) on the GPU through the C ABI
against the CPU oracle: tiny and full width, bf16 and fp32, the stream, the
one-shot and the tiled entry points, latent de-normalisation and a
checkpoint."""

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
    w = wan_synth.make_weights(base=16, seed=0, variant="wan21")
    return w, weights_dev(w)


def _bf16_check(got, ref, case):
    err, p = float(np.abs(got - ref).max()), oracle.psnr(got, ref)
    record(case, err, p)
    assert err <= TOL and p >= PSNR_MIN, (err, p)


def _clip(wv, model, z, chunk, out_dtype=torch.float32):
    B, _, T, h, w = z.shape
    st = wv.DecodeStream(model, B, h, w, max_chunk=chunk)
    v = st.decode_clip(to_dev(z), out_dtype=out_dtype)
    st.sync_status()
    return v.float().cpu().numpy()


def test_model_reports_the_variant(wv, tiny):
    model = wv.Model(tiny[1], dtype=torch.bfloat16)
    assert (model.z_dim, model.scale, model.base_dim) == (16, 8, 16)


@pytest.mark.parametrize("chunk", [1, 2])
def test_wan21_tiny_bf16(wv, tiny, chunk):
    w, wd = tiny
    z = wan_synth.make_latents((1, 16, 3, 4, 5), seed=1)
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = _clip(wv, model, z, chunk)
    assert got.shape == (1, 3, 9, 32, 40)
    _bf16_check(got, oracle.decode(oracle.round_bf16(z), rounded(w)), f"wan2.1 tiny bf16 chunk {chunk}")


def test_wan21_tiny_fp32_and_preclamp(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((2, 16, 2, 3, 4), seed=2)
    model = wv.Model(wd, dtype=torch.float32)
    st = wv.DecodeStream(model, 2, 3, 4, max_chunk=2)
    pre = torch.empty((2, 3, 5, 24, 32), device="cuda")
    out = st.decode_clip(to_dev(z), out_dtype=torch.float32, preclamp=pre)
    st.sync_status()
    ref, ref_pre = oracle.decode(z, w, return_preclamp=True)
    err = float(np.abs(out.cpu().numpy() - ref).max())
    err_pre = float(np.abs(pre.cpu().numpy() - ref_pre).max())
    record("wan2.1 tiny fp32 (clamped / pre-clamp)", max(err, err_pre), None)
    assert err <= TOL_F32 and err_pre <= TOL_F32, (err, err_pre)


def test_wan21_full_width_bf16(wv):
    w = wan_synth.make_weights(base=96, seed=0, variant="wan21")
    z = wan_synth.make_latents((1, 16, 3, 12, 12), seed=1)
    model = wv.Model(weights_dev(w), dtype=torch.bfloat16)
    got = _clip(wv, model, z, 2)
    _bf16_check(got, oracle.decode(oracle.round_bf16(z), rounded(w)), "wan2.1 full width 12x12 bf16")


def test_wan21_one_shot_and_tiled(wv, tiny):
    w, wd = tiny
    z = wan_synth.make_latents((1, 16, 2, 6, 7), seed=3)
    one = wv.decode(to_dev(z), wd, dtype=torch.bfloat16).float().cpu().numpy()
    assert one.shape == (1, 3, 5, 48, 56)
    _bf16_check(one, oracle.decode(oracle.round_bf16(z), rounded(w)), "wan2.1 tiny one-shot bf16")
    model = wv.Model(wd, dtype=torch.bfloat16)
    got = model.decode_tiled(to_dev(z), tile=(32, 32), stride=(16, 16)).float().cpu().numpy()
    ref = oracle.decode_tiled(oracle.round_bf16(z), rounded(w), tile=(32, 32), stride=(16, 16))
    _bf16_check(got, ref, "wan2.1 tiny tiled 32/16 bf16")


def test_wan21_latent_stats(wv, tiny):
    w, wd = tiny
    rng = np.random.default_rng(0)
    mean, std = rng.uniform(-1, 1, 16).astype(np.float32), rng.uniform(0.5, 3, 16).astype(np.float32)
    z = wan_synth.make_latents((1, 16, 2, 4, 4), seed=4)
    model = wv.Model(wd, dtype=torch.bfloat16)
    with pytest.raises(wv.WanError):
        model.set_latent_stats(np.zeros(48), np.ones(48))
    model.set_latent_stats(mean, std)
    got = _clip(wv, model, z, 2)
    ref = oracle.decode_normalized(z, rounded(w), mean, std, round_latents=oracle.round_bf16)
    _bf16_check(got, ref, "wan2.1 tiny bf16, de-normalised latents")


def test_wan21_checkpoint_resume(wv, tiny):
    _, wd = tiny
    z = to_dev(wan_synth.make_latents((1, 16, 4, 3, 3), seed=5))
    model = wv.Model(wd, dtype=torch.bfloat16)
    a = wv.DecodeStream(model, 1, 3, 3, max_chunk=2)
    full = a.decode_clip(z, out_dtype=torch.float32)
    b = wv.DecodeStream(model, 1, 3, 3, max_chunk=2)
    part = torch.empty_like(full)
    b.decode_chunk(z, 0, 2, part, 0)
    state = b.save_state()
    c = wv.DecodeStream(model, 1, 3, 3, max_chunk=2)
    c.load_state(state)
    c.decode_chunk(z, 2, 2, part, 5)
    torch.cuda.synchronize()
    assert torch.equal(part, full)
