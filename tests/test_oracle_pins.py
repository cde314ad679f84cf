"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one oracle function against something other than itself:
brute force on tiny inputs, a library routine (PyTorch CPU), a closed form,
or an invariant the page "wan22_vae_decode/reference.py" states.  Chosen so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import wan_synth

RNG = np.random.default_rng(1234)


def _rand(*shape):
    return RNG.standard_normal(shape).astype(np.float32)


# ----------------------------------------------------------------- causal conv
def brute_causal_conv(x, w, b, history):
    """Direct convolution in fp64 with explicit loops (7 nested).

    Time index t + dt - 2*(kt//2) relative to x's first frame: negative indices
    read the history from its end, missing history reads zero; space is zero
    padded by kh//2, kw//2.
    """
    B, Ci, T, H, W = x.shape
    Co, _, kt, kh, kw = w.shape
    front = 2 * (kt // 2)
    nh = 0 if history is None else history.shape[2]
    out = np.zeros((B, Co, T, H, W))
    for bb in range(B):
        for o in range(Co):
            for t in range(T):
                for y in range(H):
                    for xx in range(W):
                        s = float(b[o])
                        for c in range(Ci):
                            for dt in range(kt):
                                ts = t + dt - front
                                if ts >= 0:
                                    frame = x[bb, c, ts]
                                elif -ts <= nh:
                                    frame = history[bb, c, nh + ts]
                                else:
                                    continue
                                for dy in range(kh):
                                    ys = y + dy - kh // 2
                                    if not 0 <= ys < H:
                                        continue
                                    for dx in range(kw):
                                        xs = xx + dx - kw // 2
                                        if 0 <= xs < W:
                                            s += float(w[o, c, dt, dy, dx]) * float(frame[ys, xs])
                        out[bb, o, t, y, xx] = s
    return out


@pytest.mark.parametrize("kernel", [(3, 3, 3), (3, 1, 1), (1, 1, 1), (1, 3, 3)])
@pytest.mark.parametrize("nhist", [None, 1, 2])
def test_causal_conv_brute_force(kernel, nhist):
    x = _rand(1, 3, 2, 4, 5)
    w = _rand(2, 3, *kernel)
    b = _rand(2)
    hist = None if nhist is None else _rand(1, 3, nhist, 4, 5)
    got = oracle.causal_conv(x, w, b, hist)
    want = brute_causal_conv(x, w, b, hist)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("nhist", [None, 1, 2])
def test_causal_conv_vs_torch_conv3d(nhist):
    """The same conv through torch's conv3d on explicitly padded input."""
    x = _rand(2, 8, 3, 6, 7)
    w = _rand(5, 8, 3, 3, 3)
    b = _rand(5)
    hist = None if nhist is None else _rand(2, 8, nhist, 6, 7)
    seq = x if hist is None else np.concatenate([hist, x], axis=2)
    zeros = 2 - (0 if hist is None else nhist)
    xp = torch.from_numpy(seq).double()
    xp = F.pad(xp, (1, 1, 1, 1, zeros, 0))
    want = F.conv3d(xp, torch.from_numpy(w).double(), torch.from_numpy(b).double()).numpy()
    got = oracle.causal_conv(x, w, b, hist)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5)


def test_conv2d_vs_torch():
    x = _rand(1, 4, 2, 5, 6)
    w = _rand(3, 4, 3, 3)
    b = _rand(3)
    got = oracle.conv2d(x, w, b)
    for t in range(2):
        want = F.conv2d(torch.from_numpy(x[:, :, t]).double(), torch.from_numpy(w).double(),
                        torch.from_numpy(b).double(), padding=1).numpy()
        np.testing.assert_allclose(got[:, :, t], want, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("chunk", [1, 2])
def test_cached_conv_frame_loop_equals_whole_sequence(chunk):
    """Section "Causal caches": the chunk loop with caches computes what one
    causal conv over the whole sequence (zeros before frame 0) computes."""
    from oracle.wan_decode import cached_conv
    x = _rand(1, 4, 5, 3, 4)
    wts = {"c.weight": _rand(3, 4, 3, 3, 3), "c.bias": _rand(3)}
    whole = oracle.causal_conv(x, wts["c.weight"], wts["c.bias"])
    cache = {}
    parts = [cached_conv(x[:, :, i:i + chunk], wts, "c", cache) for i in range(0, 5, chunk)]
    np.testing.assert_allclose(np.concatenate(parts, axis=2), whole, rtol=1e-5, atol=1e-5)
    # after the loop the cache holds the last two input frames
    np.testing.assert_array_equal(cache["c"], x[:, :, -2:])


def test_cache_after_one_frame_chunks():
    """After a one-frame chunk the cache holds the previous last frame and this one."""
    from oracle.wan_decode import cached_conv
    x = _rand(1, 2, 3, 2, 2)
    wts = {"c.weight": _rand(2, 2, 3, 1, 1), "c.bias": _rand(2)}
    cache = {}
    cached_conv(x[:, :, 0:1], wts, "c", cache)
    assert cache["c"].shape[2] == 1
    np.testing.assert_array_equal(cache["c"][:, :, 0], x[:, :, 0])
    cached_conv(x[:, :, 1:2], wts, "c", cache)
    np.testing.assert_array_equal(cache["c"], x[:, :, 0:2])
    cached_conv(x[:, :, 2:3], wts, "c", cache)
    np.testing.assert_array_equal(cache["c"], x[:, :, 1:3])


# -------------------------------------------------------------------- RMS norm
def test_rms_norm_length_is_sqrt_c():
    x = _rand(2, 16, 3, 4, 5)
    g = 1 + 0.1 * _rand(16)
    y = oracle.rms_norm(x, g)
    ratio = y / g.reshape(1, 16, 1, 1, 1)
    np.testing.assert_allclose(np.linalg.norm(ratio.astype(np.float64), axis=1), math.sqrt(16), rtol=1e-6)


def test_rms_norm_uniform_gamma_and_zero_and_scale():
    x = _rand(1, 9, 2, 3, 3)
    y = oracle.rms_norm(x, np.full(9, -2.5, np.float32))
    np.testing.assert_allclose(np.linalg.norm(y.astype(np.float64), axis=1), 3.0 * 2.5, rtol=1e-6)
    # x = 0: the max(., 1e-12) branch gives 0, not NaN
    z = oracle.rms_norm(np.zeros((1, 4, 1, 2, 2), np.float32), np.ones(4, np.float32))
    assert np.all(z == 0)
    # invariant to positive scaling of x
    g = 1 + 0.1 * _rand(9)
    np.testing.assert_allclose(oracle.rms_norm(7.0 * x, g), oracle.rms_norm(x, g), rtol=1e-5, atol=1e-6)


def test_rms_norm_vs_torch_normalize():
    x = _rand(2, 32, 2, 3, 4)
    g = 1 + 0.1 * _rand(32)
    want = (F.normalize(torch.from_numpy(x).double(), dim=1) * math.sqrt(32)
            * torch.from_numpy(g).double().view(1, 32, 1, 1, 1)).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g), want, rtol=1e-5, atol=1e-6)


# -------------------------------------------------------------------- attention
def _attn_weights(C):
    return {
        "a.norm.gamma": 1 + 0.1 * _rand(C),
        "a.to_qkv.weight": _rand(3 * C, C, 1, 1) / math.sqrt(C),
        "a.to_qkv.bias": 0.1 * _rand(3 * C),
        "a.proj.weight": _rand(C, C, 1, 1) / math.sqrt(C),
        "a.proj.bias": 0.1 * _rand(C),
    }


def _proj_v_plus_x(x, w, C):
    n = oracle.rms_norm(x, w["a.norm.gamma"])
    qkv = oracle.conv2d(n, w["a.to_qkv.weight"], w["a.to_qkv.bias"])
    return oracle.conv2d(qkv[:, 2 * C:], w["a.proj.weight"], w["a.proj.bias"]) + x


def test_attention_one_key_returns_v():
    """Page "Fix the Wan VAE attention block": softmax over a single key is 1,
    so with h*w = 1 the block computes proj(v) + x exactly."""
    C = 8
    w = _attn_weights(C)
    x = _rand(2, C, 3, 1, 1)
    np.testing.assert_allclose(oracle.attention(x, w, "a"), _proj_v_plus_x(x, w, C), rtol=1e-5, atol=1e-5)


def test_attention_many_keys_differs_from_v():
    """With distinct positions the attention mixes them: not proj(v) + x."""
    C = 8
    w = _attn_weights(C)
    x = _rand(1, C, 2, 4, 6)
    diff = np.abs(oracle.attention(x, w, "a") - _proj_v_plus_x(x, w, C)).max()
    assert diff > 1e-2


def test_attention_vs_torch_sdpa_and_permutation():
    C, H, W = 16, 3, 5
    w = _attn_weights(C)
    x = _rand(1, C, 2, H, W)
    got = oracle.attention(x, w, "a")
    # torch composition: normalize, 1x1 conv, sdpa (one head), 1x1 conv, + x
    xt = torch.from_numpy(x).double()
    for t in range(2):
        f = xt[:, :, t]
        n = F.normalize(f, dim=1) * math.sqrt(C) * torch.from_numpy(w["a.norm.gamma"]).double().view(1, C, 1, 1)
        qkv = F.conv2d(n, torch.from_numpy(w["a.to_qkv.weight"]).double(), torch.from_numpy(w["a.to_qkv.bias"]).double())
        seq = qkv.flatten(2).transpose(1, 2)                       # [1, HW, 3C]
        q, k, v = seq[..., :C], seq[..., C:2 * C], seq[..., 2 * C:]
        o = F.scaled_dot_product_attention(q[:, None], k[:, None], v[:, None])[:, 0]   # [1, HW, C]
        o = o.transpose(1, 2).reshape(1, C, H, W)
        y = F.conv2d(o, torch.from_numpy(w["a.proj.weight"]).double(), torch.from_numpy(w["a.proj.bias"]).double()) + f
        np.testing.assert_allclose(got[:, :, t], y.numpy(), rtol=1e-4, atol=1e-5)
    # permuting the positions of a frame permutes the outputs the same way
    perm = RNG.permutation(H * W)
    xp = x.reshape(1, C, 2, H * W)[..., perm].reshape(1, C, 2, H, W)
    gp = oracle.attention(xp, w, "a")
    np.testing.assert_allclose(gp, got.reshape(1, C, 2, H * W)[..., perm].reshape(1, C, 2, H, W), rtol=1e-4, atol=1e-5)


def test_softmax_rows_brute():
    s = _rand(4, 7).astype(np.float64) * 5
    p = oracle.wan_decode.softmax_rows(s)
    for r in range(4):
        e = [math.exp(v) for v in s[r]]
        tot = sum(e)
        np.testing.assert_allclose(p[r], [v / tot for v in e], rtol=1e-12)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-12)


# ---------------------------------------------------------------- reshuffles
def test_time_interleave_brute():
    C, T = 3, 4
    y = np.arange(1 * 2 * C * T * 2 * 3, dtype=np.float32).reshape(1, 2 * C, T, 2, 3)
    out = oracle.time_interleave(y)
    assert out.shape == (1, C, 2 * T, 2, 3)
    for c in range(C):
        for t in range(T):
            np.testing.assert_array_equal(out[0, c, 2 * t], y[0, c, t])
            np.testing.assert_array_equal(out[0, c, 2 * t + 1], y[0, C + c, t])


def test_time_upsample_selector_weights():
    """A time conv whose weights pick input channel c into output c and the
    negated channel into output C + c: frame 2t holds +x, frame 2t + 1 holds -x."""
    from oracle.wan_decode import time_upsample
    C = 3
    x = _rand(1, C, 2, 2, 2)
    w = np.zeros((2 * C, C, 3, 1, 1), np.float32)
    for c in range(C):
        w[c, c, 2] = 1.0
        w[C + c, c, 2] = -1.0
    out = time_upsample(x, {"t.weight": w, "t.bias": np.zeros(2 * C, np.float32)}, "t", {})
    np.testing.assert_array_equal(out[:, :, 0::2], x)
    np.testing.assert_array_equal(out[:, :, 1::2], -x)


def test_nearest_exact_vs_repeat_and_torch():
    x = _rand(2, 3, 4, 5)
    up = oracle.nearest_exact_up2(x)
    np.testing.assert_array_equal(up, x.repeat(2, axis=-2).repeat(2, axis=-1))
    want = F.interpolate(torch.from_numpy(x), scale_factor=(2.0, 2.0), mode="nearest-exact").numpy()
    np.testing.assert_array_equal(up, want)


def test_dup_up_r8_is_nearest_x2_in_t_h_w():
    x = _rand(1, 4, 3, 2, 3)
    d = oracle.dup_up(x, 4, 2, first=False)   # r = 4*2*4/4 = 8
    want = x.repeat(2, axis=2).repeat(2, axis=3).repeat(2, axis=4)
    np.testing.assert_array_equal(d, want)
    # first chunk: only the last of the two time copies
    np.testing.assert_array_equal(oracle.dup_up(x, 4, 2, first=True), want[:, :, 1:])


def test_dup_up_r2_channel_pairs_to_rows():
    x = np.arange(1 * 8 * 2 * 2 * 3, dtype=np.float32).reshape(1, 8, 2, 2, 3)
    d = oracle.dup_up(x, 4, 1, first=False)   # r = 4*1*4/8 = 2
    assert d.shape == (1, 4, 2, 4, 6)
    for c, t, y, xx, i, j in itertools.product(range(4), range(2), range(2), range(3), range(2), range(2)):
        assert d[0, c, t, 2 * y + i, 2 * xx + j] == x[0, 2 * c + i, t, y, xx]


def test_dup_up_index_formula_brute():
    cin, cout, ft = 6, 3, 2          # r = 3*2*4/6 = 4
    x = np.arange(1 * cin * 2 * 2 * 2, dtype=np.float32).reshape(1, cin, 2, 2, 2)
    d = oracle.dup_up(x, cout, ft, first=False)
    r = cout * ft * 4 // cin
    for c, t, a, y, i, xx, j in itertools.product(range(cout), range(2), range(ft), range(2), range(2), range(2), range(2)):
        assert d[0, c, ft * t + a, 2 * y + i, 2 * xx + j] == x[0, (4 * ft * c + 4 * a + 2 * i + j) // r, t, y, xx]


def test_unpatchify_bijection_and_formula():
    out = np.arange(2 * 12 * 3 * 2 * 4, dtype=np.float32).reshape(2, 12, 3, 2, 4)
    v = oracle.unpatchify(out)
    assert v.shape == (2, 3, 3, 4, 8)
    np.testing.assert_array_equal(np.sort(v.ravel()), out.ravel())
    for b, k, f, y, xx, i, j in itertools.product(range(2), range(3), range(3), range(2), range(4), range(2), range(2)):
        assert v[b, k, f, 2 * y + i, 2 * xx + j] == out[b, 4 * k + 2 * j + i, f, y, xx]
    # the inverse (patchify) written directly from the formula round-trips
    back = np.empty_like(out)
    for k, i, j in itertools.product(range(3), range(2), range(2)):
        back[:, 4 * k + 2 * j + i] = v[:, k, :, i::2, j::2]
    np.testing.assert_array_equal(back, out)


def test_round_bf16_ties_and_vs_torch():
    vals = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 3.0e-39, 65504.0], np.float32)
    r = oracle.round_bf16(vals)
    assert r[0] == 1.0 and r[1] == 1.0 and r[2] == 1 + 2 ** -6 and r[3] == -1.0
    x = (_rand(10000) * 10.0 ** RNG.integers(-20, 20, 10000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x), want)


def test_psnr_closed_form():
    a = _rand(1000).astype(np.float64).clip(-0.9, 0.9)
    assert math.isclose(oracle.psnr(a, a + 0.02), 10 * math.log10(1 / 0.01 ** 2), rel_tol=1e-9)
    assert oracle.psnr(a, a) == float("inf")


# ------------------------------------------------------------- whole decoder
def test_frame_count_4t_minus_3(tiny_weights):
    for T in (1, 2, 3, 4):
        z = wan_synth.make_latents((1, 48, T, 2, 2), seed=10 + T)
        v = oracle.decode(z, tiny_weights)
        assert v.shape == (1, 3, 4 * T - 3, 32, 32)
        assert np.all(np.abs(v) <= 1.0)


def test_frame_loop_equals_whole_sequence(tiny_weights):
    """Section "Causal caches": the frame loop equals the whole-sequence form up
    to rounding (the page reports max 1.7e-5 in fp32 on trained weights)."""
    z = wan_synth.make_latents((1, 48, 3, 4, 4), seed=1)
    _, f1 = oracle.decode(z, tiny_weights, chunk=1, return_preclamp=True)
    _, f2 = oracle.decode_whole(z, tiny_weights, return_preclamp=True)
    _, f3 = oracle.decode(z, tiny_weights, chunk=2, return_preclamp=True)
    scale = np.abs(f2).max()
    assert np.abs(f1 - f2).max() <= 1e-4 * scale
    assert np.abs(f3 - f2).max() <= 1e-4 * scale


def test_causality(tiny_weights):
    """Output frames < 4k-3 depend only on latent frames < k (frame loop)."""
    z = wan_synth.make_latents((1, 48, 3, 3, 3), seed=7)
    v = oracle.decode(z, tiny_weights)
    z2 = z.copy()
    z2[:, :, 2:] += 1.0
    v2 = oracle.decode(z2, tiny_weights)
    k = 2
    np.testing.assert_array_equal(v[:, :, :4 * k - 3], v2[:, :, :4 * k - 3])
    assert np.abs(v[:, :, 4 * k - 3:] - v2[:, :, 4 * k - 3:]).max() > 1e-3


def test_batch_independence(tiny_weights):
    z = wan_synth.make_latents((2, 48, 2, 3, 2), seed=8)
    both = oracle.decode(z, tiny_weights)
    for b in range(2):
        one = oracle.decode(z[b:b + 1], tiny_weights)
        np.testing.assert_allclose(both[b:b + 1], one, rtol=0, atol=2e-6)


def test_decode_ignores_foreign_names(tiny_weights):
    w = dict(tiny_weights)
    w["encoder.conv_in.weight"] = np.full((3, 3), np.nan, np.float32)
    w["quant_conv.weight"] = np.full((3, 3), np.nan, np.float32)
    z = wan_synth.make_latents((1, 48, 1, 2, 2), seed=9)
    np.testing.assert_array_equal(oracle.decode(z, w), oracle.decode(z, tiny_weights))


def test_oracle_vs_independent_torch_composition(tiny_weights):
    """The oracle's frame loop against a separately written whole-sequence
    decode built from torch library ops in fp64 (tests/torch_composition.py)."""
    from tests.torch_composition import decode_whole_torch
    z = wan_synth.make_latents((1, 48, 3, 4, 4), seed=1)
    _, pre = oracle.decode(z, tiny_weights, return_preclamp=True)
    want = decode_whole_torch(z, tiny_weights)
    assert want.shape == pre.shape
    assert np.abs(pre - want).max() <= 1e-4 * np.abs(want).max()
