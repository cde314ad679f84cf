"""The Wan2.2-TI2V-5B VAE decode, written out plainly in NumPy (CPU oracle),
and the Wan2.1 VAE decode that shares its parts.

Test infrastructure only: the CUDA path never imports this module.

Source: the page "wan22_vae_decode/reference.py" (FastVideo), a standalone
description of diffusers' ``AutoencoderKLWan._decode`` for the TI2V-5B VAE.
Each function below cites the docstring section or function of that page whose
definition it writes out.  Layout is the page's: [B, C, T, H, W] (NCDHW).

Precision: activations are fp32; convolutions are sums over kernel taps of
fp32 BLAS matmuls; the RMS norm's vector length and the softmax's exponentials
and sums are taken in fp64.  A bf16 decode is represented by feeding the oracle
bf16-rounded latents and weights (``round_bf16``), the first step of the
page's bf16 contract (section "Precision"); the oracle itself always computes
in fp32.

Wan2.1 VAE (``AutoencoderKLWan`` of the Wan 2.1 and Wan 2.2 A14B pipelines,
page "Fix the Wan VAE attention block"): the page fixes z_dim 16, 8x spatial
compression (720p latents of 90x160, attention over 14,400 positions per
frame) and that its attention block is the same one-head block over a
frame's positions.  The rest of its decoder is not on the pages; the reading
taken here is that model's published configuration, built from the same
parts: base dim 96, channel multipliers (1, 2, 4, 4), two residual blocks
per level (three per up block), temporal upsampling in the first two up
blocks, and resamplers whose conv halves the channels (C -> C/2) with no
DupUp3D shortcut and no 2x2 patching; conv_out writes the 3 colours
directly.  Its up blocks, for base dim b: 4b -> 4b (time and space), 2b ->
4b (time and space), 2b -> 2b (space), b -> b; parameter names as in
diffusers (``upsamplers.0.time_conv``, ``upsamplers.0.resample.1``).  The
variant is read from the weights: post_quant_conv 16 -> 16 is Wan2.1.
"""

from __future__ import annotations

import math

import numpy as np

# Frames of history kept by a causal conv with a 3-frame kernel (section
# "Causal caches": the last two frames of its input).
CACHE_T = 2
# unpatchify's patch edge (section "What is computed", item 3).
PATCH_SIZE = 2
# Parameter-name prefixes that decode uses (function ``decode``).
PREFIXES = ("decoder.", "post_quant_conv.")
RESNETS_PER_UP_BLOCK = 3
F32 = np.float32


def round_bf16(x) -> np.ndarray:
    """fp32 -> nearest bf16 value (round to nearest, ties to even), as fp32.

    Section "Precision": a bf16 decode starts from the latents and weights
    rounded to bf16.  bf16 keeps the top 16 bits of an IEEE fp32 word; the
    dropped low 16 bits round the kept part to nearest, ties to even.
    """
    a = np.ascontiguousarray(x, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)
    return rounded.astype(np.uint32).view(np.float32).reshape(a.shape)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x)) (``residual_block``)."""
    x = np.asarray(x, dtype=F32)
    with np.errstate(over="ignore"):
        return (x / (F32(1.0) + np.exp(-x))).astype(F32)


def rms_norm(x: np.ndarray, gamma: np.ndarray) -> np.ndarray:
    """WanRMS_norm over the channel axis (axis 1).

    Section "What is computed", "The parts", second bullet: F.normalize, i.e.
    x / max(||x||_2, 1e-12) over channels, times sqrt(C), times gamma (one
    value per channel, no bias).
    """
    x = np.asarray(x, dtype=F32)
    C = x.shape[1]
    length = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=1, keepdims=True))
    unit = x.astype(np.float64) / np.maximum(length, 1e-12)
    g = np.asarray(gamma, dtype=np.float64).reshape((1, C) + (1,) * (x.ndim - 2))
    return (unit * math.sqrt(C) * g).astype(F32)


def causal_conv(x: np.ndarray, weight: np.ndarray, bias: np.ndarray, history=None) -> np.ndarray:
    """WanCausalConv3d on x [B, Ci, t, h, w] (``causal_conv``).

    "The parts", first bullet: stride 1; zero padding of kh//2 and kw//2 on
    both sides in space; in time 2*(kt//2) frames before x and none after:
    the conv's history frames (the latest ones), zeros for the frames the
    history lacks.  Then

        out[b,o,t,y,x] = bias[o]
            + sum_{c,dt,dy,dx} W[o,c,dt,dy,dx] * xpad[b,c,t+dt,y+dy,x+dx],

    evaluated as a sum over the kt*kh*kw taps of [N, Ci] @ [Ci, Co] matmuls.
    """
    x = np.asarray(x, dtype=F32)
    weight = np.asarray(weight, dtype=F32)
    B, Ci, T, H, W = x.shape
    Co, wci, kt, kh, kw = weight.shape
    assert wci == Ci, (weight.shape, x.shape)
    front = 2 * (kt // 2)
    if history is not None and front > 0 and history.shape[2] > 0:
        hist = np.asarray(history, dtype=F32)[:, :, -front:]
        x = np.concatenate([hist, x], axis=2)
        front -= hist.shape[2]
    xp = np.pad(x, ((0, 0), (0, 0), (front, 0), (kh // 2, kh // 2), (kw // 2, kw // 2)))
    xcl = np.ascontiguousarray(xp.transpose(0, 2, 3, 4, 1))  # [B, Tp, Hp, Wp, Ci]
    acc = np.zeros((B * T * H * W, Co), dtype=F32)
    tmp = np.empty_like(acc)
    for dt in range(kt):
        for dy in range(kh):
            for dx in range(kw):
                slab = xcl[:, dt:dt + T, dy:dy + H, dx:dx + W, :].reshape(-1, Ci)
                np.matmul(slab, np.ascontiguousarray(weight[:, :, dt, dy, dx].T), out=tmp)
                acc += tmp
    acc += np.asarray(bias, dtype=F32)[None, :]
    return np.ascontiguousarray(acc.reshape(B, T, H, W, Co).transpose(0, 4, 1, 2, 3))


def conv2d(x: np.ndarray, weight: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Per-frame conv2d of x [B, Ci, t, h, w] with weight [Co, Ci, kh, kw].

    Zero padding kh//2, kw//2 (1 for the 3x3 resample conv, 0 for the 1x1
    attention convs): the causal conv above with a one-frame kernel.
    """
    return causal_conv(x, np.asarray(weight)[:, :, None], bias)


def cached_conv(x, weights, name, cache):
    """A 3-frame causal conv of one chunk with its history (section "Causal caches").

    The conv sees cache[name] before x; afterwards cache[name] holds the last
    CACHE_T frames of what it convolved (history followed by x): after a
    one-frame chunk, the previous chunk's last frame and this one.
    """
    history = cache.get(name)
    out = causal_conv(x, weights[f"{name}.weight"], weights[f"{name}.bias"], history)
    seen = x if history is None else np.concatenate([history, x], axis=2)
    cache[name] = np.ascontiguousarray(seen[:, :, -CACHE_T:])
    return out


def residual_block(x, weights, name, cache):
    """WanResidualBlock ("The parts", third bullet; ``residual_block``).

    x1 = conv1(SiLU(norm1(x))), x2 = conv2(SiLU(norm2(x1))); returns
    x2 + shortcut, the shortcut being x or a 1x1x1 conv of x when the channel
    counts differ.
    """
    if f"{name}.conv_shortcut.weight" in weights:
        shortcut = causal_conv(x, weights[f"{name}.conv_shortcut.weight"], weights[f"{name}.conv_shortcut.bias"])
    else:
        shortcut = x
    h = cached_conv(silu(rms_norm(x, weights[f"{name}.norm1.gamma"])), weights, f"{name}.conv1", cache)
    h = cached_conv(silu(rms_norm(h, weights[f"{name}.norm2.gamma"])), weights, f"{name}.conv2", cache)
    return (h + shortcut).astype(F32)


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax in fp64: subtract the row maximum, exponentiate, normalise."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def attention(x, weights, name):
    """WanAttentionBlock, per frame ("The parts", fourth bullet; ``attention``).

    n = RMS norm of the frame; q, k, v = channels [0,C), [C,2C), [2C,3C) of a
    1x1 conv C -> 3C of n; one head: softmax(q k^T / sqrt(C)) v over the h*w
    positions (no mask); a 1x1 conv C -> C; plus x.
    """
    x = np.asarray(x, dtype=F32)
    B, C, T, H, W = x.shape
    wqkv = np.asarray(weights[f"{name}.to_qkv.weight"], dtype=F32).reshape(3 * C, C)
    bqkv = np.asarray(weights[f"{name}.to_qkv.bias"], dtype=F32)
    wp = np.asarray(weights[f"{name}.proj.weight"], dtype=F32).reshape(C, C)
    bp = np.asarray(weights[f"{name}.proj.bias"], dtype=F32)
    gamma = weights[f"{name}.norm.gamma"]
    out = np.empty_like(x)
    for b in range(B):
        for t in range(T):
            frame = x[b, :, t]                                  # [C, H, W]
            n = rms_norm(frame[None], gamma)[0].reshape(C, H * W)
            qkv = wqkv @ n + bqkv[:, None]                      # [3C, HW]
            q, k, v = qkv[:C], qkv[C:2 * C], qkv[2 * C:]
            scores = (q.T @ k) / F32(math.sqrt(C))              # [HW queries, HW keys]
            p = softmax_rows(scores)
            o = (p @ v.T.astype(np.float64)).astype(F32)        # [HW, C]
            y = wp @ o.T + bp[:, None]                          # [C, HW]
            out[b, :, t] = y.reshape(C, H, W) + frame
    return out


def time_interleave(y: np.ndarray) -> np.ndarray:
    """[B, 2C, t, h, w] -> [B, C, 2t, h, w]: channel c becomes frame 2t and
    channel C + c frame 2t + 1 ("The parts", fifth bullet, upsample3d)."""
    B, C2, T, H, W = y.shape
    C = C2 // 2
    out = np.empty((B, C, 2 * T, H, W), dtype=y.dtype)
    for t in range(T):
        out[:, :, 2 * t] = y[:, :C, t]
        out[:, :, 2 * t + 1] = y[:, C:, t]
    return out


def time_upsample(x, weights, name, cache):
    """upsample3d's time conv: causal 3x1x1 conv C -> 2C, then the interleave
    (``time_upsample``)."""
    return time_interleave(cached_conv(x, weights, name, cache))


def nearest_exact_up2(x: np.ndarray) -> np.ndarray:
    """Nearest-exact x2 in the last two axes (WanUpsample, mode nearest-exact).

    nearest-exact maps output index d to source index floor((d + 0.5) * in/out);
    it only copies values.
    """
    H, W = x.shape[-2:]
    ys = np.floor((np.arange(2 * H) + 0.5) * (H / (2 * H))).astype(np.int64)
    xs = np.floor((np.arange(2 * W) + 0.5) * (W / (2 * W))).astype(np.int64)
    return x[..., ys[:, None], xs[None, :]]


def spatial_upsample(x, weights, name):
    """upsample2d: per frame, nearest x2 in h and w, then a 3x3 conv2d C -> C
    (C -> C/2 in the Wan2.1 decoder) with zero padding 1 (``spatial_upsample``)."""
    return conv2d(nearest_exact_up2(x), weights[f"{name}.weight"], weights[f"{name}.bias"])


def dup_up(x: np.ndarray, out_channels: int, ft: int, first: bool) -> np.ndarray:
    """DupUp3D ("The parts", sixth bullet; ``dup_up``).

    Each input channel is repeated r = out*ft*4/in times over the (ft, 2, 2)
    sub-positions: dup[c, ft*t + a, 2y + i, 2x + j] = x[(4*ft*c + 4a + 2i + j)//r, t, y, x].
    On the first chunk only the last of the ft copies in time is kept.
    """
    B, Cin, T, H, W = x.shape
    r = out_channels * ft * 4 // Cin
    out = np.empty((B, out_channels, ft * T, 2 * H, 2 * W), dtype=x.dtype)
    c = np.arange(out_channels)
    for a in range(ft):
        for i in range(2):
            for j in range(2):
                src = (4 * ft * c + 4 * a + 2 * i + j) // r
                out[:, :, a::ft, i::2, j::2] = x[:, src]
    return out[:, :, ft - 1:] if first else out


def up_block(x, weights, i, cache, first, up_blocks, wan21: bool = False):
    """WanResidualUpBlock i (``up_block``): three residual blocks, then for up
    blocks 0-2 the resampler plus DupUp3D of the block's input.  In the Wan2.1
    decoder the resampler (``upsamplers.0``) halves the channels and there is
    no DupUp3D.

    Section "The first latent frame yields one frame": on the first chunk the
    time conv is skipped for its first frame, which passes through as one
    frame; the time conv's input sequence begins with the second latent frame.
    """
    _, cout, temporal, spatial = up_blocks[i]
    name = f"decoder.up_blocks.{i}"
    ups = f"{name}.upsamplers.0" if wan21 else f"{name}.upsampler"
    block_input = x
    for j in range(RESNETS_PER_UP_BLOCK):
        x = residual_block(x, weights, f"{name}.resnets.{j}", cache)
    if not spatial:
        return x
    if temporal:
        tconv = f"{ups}.time_conv"
        if first:
            rest = x[:, :, 1:]
            if rest.shape[2] > 0:
                x = np.concatenate([x[:, :, :1], time_upsample(rest, weights, tconv, cache)], axis=2)
            else:
                x = x[:, :, :1]
        else:
            x = time_upsample(x, weights, tconv, cache)
    x = spatial_upsample(x, weights, f"{ups}.resample.1")
    if wan21:
        return x
    return (x + dup_up(block_input, cout, 2 if temporal else 1, first)).astype(F32)


def _up_blocks(base: int):
    """Section "What is computed": (in, out, temporal, spatial) per up block,
    channels 4b/4b, 4b/4b, 4b/2b, 2b/b for decoder base dim b."""
    return ((4 * base, 4 * base, True, True), (4 * base, 4 * base, True, True),
            (4 * base, 2 * base, False, True), (2 * base, base, False, False))


def _up_blocks_wan21(base: int):
    """The Wan2.1 decoder's (in, out, temporal, spatial) per up block; each
    resampler halves its block's output channels, so the next block starts
    from half of them."""
    return ((4 * base, 4 * base, True, True), (2 * base, 4 * base, True, True),
            (2 * base, 2 * base, False, True), (base, base, False, False))


def is_wan21(weights) -> bool:
    """The Wan2.1 VAE (z_dim 16) rather than TI2V-5B's (z_dim 48)."""
    return np.asarray(weights["post_quant_conv.weight"]).shape[0] == 16


def decode_chunk(x, weights, cache, first):
    """The decoder on a chunk of latent frames x [B, 48, n, h, w] (``decode_chunk``).

    conv_in, mid block (residual, attention, residual), up blocks 0-3, then
    norm_out, SiLU and conv_out.  Returns [B, 12, 4n-3 (first) or 4n, 8h, 8w]
    (Wan2.1: x [B, 16, n, h, w] -> [B, 3, ..., 8h, 8w]).
    """
    base = np.asarray(weights["decoder.conv_in.weight"]).shape[0] // 4
    wan21 = is_wan21(weights)
    ups = _up_blocks_wan21(base) if wan21 else _up_blocks(base)
    x = cached_conv(x, weights, "decoder.conv_in", cache)
    x = residual_block(x, weights, "decoder.mid_block.resnets.0", cache)
    x = attention(x, weights, "decoder.mid_block.attentions.0")
    x = residual_block(x, weights, "decoder.mid_block.resnets.1", cache)
    for i in range(len(ups)):
        x = up_block(x, weights, i, cache, first, ups, wan21)
    x = silu(rms_norm(x, weights["decoder.norm_out.gamma"]))
    return cached_conv(x, weights, "decoder.conv_out", cache)


def unpatchify(out: np.ndarray, p: int = PATCH_SIZE) -> np.ndarray:
    """[B, 3*p*p, F, h, w] -> [B, 3, F, p*h, p*w] (section "What is computed", 3):
    video[b, k, f, p*y + i, p*x + j] = out[b, (k*p + j)*p + i, f, y, x]."""
    B, CP, Fr, H, W = out.shape
    K = CP // (p * p)
    video = np.empty((B, K, Fr, p * H, p * W), dtype=out.dtype)
    for i in range(p):
        for j in range(p):
            video[:, :, :, i::p, j::p] = out[:, [(k * p + j) * p + i for k in range(K)]]
    return video


def decode(z, weights, chunk: int = 1, return_preclamp: bool = False):
    """decode(z, weights): latents [B, 48, T, h, w] -> video [B, 3, 4T-3, 16h, 16w]
    in [-1, 1] (function ``decode``; section "What is computed", items 1-4).
    Wan2.1 weights: latents [B, 16, T, h, w] -> video [B, 3, 4T-3, 8h, 8w],
    no unpatchify.

    post_quant_conv over all T frames at once, then the decoder chunk by chunk
    (``chunk`` latent frames per call, 1 being the page's frame loop) with the
    causal caches carried between chunks, the chunks concatenated on time,
    unpatchify, clamp.  With ``return_preclamp`` the unclamped video is
    returned as well.
    """
    w = {k: v for k, v in weights.items() if k.startswith(PREFIXES)}
    x = causal_conv(z, w["post_quant_conv.weight"], w["post_quant_conv.bias"])
    T = x.shape[2]
    cache: dict = {}
    outs = [decode_chunk(x[:, :, i:i + chunk], w, cache, first=(i == 0)) for i in range(0, T, chunk)]
    out = np.concatenate(outs, axis=2)
    video = out if is_wan21(w) else unpatchify(out)
    clamped = np.clip(video, -1.0, 1.0).astype(F32)
    return (clamped, video) if return_preclamp else clamped


def decode_whole(z, weights, return_preclamp: bool = False):
    """The whole-sequence form (section "Causal caches", last sentences): every
    causal conv over all frames of its level with two zero frames before the
    first, the time conv over the frames after the first, DupUp3D doubling
    every frame but the first.  It is the decoder run on all frames as one
    first chunk with empty caches."""
    return decode(z, weights, chunk=np.asarray(z).shape[2], return_preclamp=return_preclamp)


def psnr(a, b) -> float:
    """PSNR of two signals in [-1, 1]: 10*log10(1 / mean(((a - b)/2)^2)), fp64
    (page "Fix the Wan VAE attention block", comparison script)."""
    d = (np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)) / 2.0
    mse = float(np.mean(d * d))
    return float("inf") if mse == 0.0 else 10.0 * math.log10(1.0 / mse)
