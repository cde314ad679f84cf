"""A second, test-only CPU implementation of the decode, in PyTorch fp64.

Written independently of ``oracle`` and in the other form the page
"wan22_vae_decode/reference.py" (section "Causal caches") gives: the
whole sequence at once, every causal conv over all frames of its level with
two zero frames in front, the time conv over the frames after the first,
DupUp3D doubling every frame but the first.  Built from torch library ops
(conv3d/conv2d, normalize, silu, scaled_dot_product_attention, interpolate)
so that a composition slip in the oracle (a misplaced norm, a wrong shortcut,
a swapped resampler order) shows up as a disagreement.  Wan2.1 weights
(post_quant_conv 16 -> 16): resamplers under ``upsamplers.0`` that halve the
channels, no DupUp3D shortcut, conv_out giving the 3 colours directly.
"""

import math

import numpy as np
import torch
import torch.nn.functional as F


def decode_whole_torch(z, weights):
    w = {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in weights.items()
         if k.startswith(("decoder.", "post_quant_conv."))}

    def cconv(x, name):
        k = w[f"{name}.weight"]
        kt, kh, kw = k.shape[2:]
        return F.conv3d(F.pad(x, (kw // 2, kw // 2, kh // 2, kh // 2, 2 * (kt // 2), 0)), k, w[f"{name}.bias"])

    def norm(x, name):
        g = w[f"{name}.gamma"].reshape(1, -1, *([1] * (x.dim() - 2)))
        return F.normalize(x, dim=1) * math.sqrt(x.shape[1]) * g

    def resnet(x, name):
        sc = cconv(x, f"{name}.conv_shortcut") if f"{name}.conv_shortcut.weight" in w else x
        h = cconv(F.silu(norm(x, f"{name}.norm1")), f"{name}.conv1")
        h = cconv(F.silu(norm(h, f"{name}.norm2")), f"{name}.conv2")
        return h + sc

    def attn(x, name):
        B, C, T, H, W = x.shape
        f = x.permute(0, 2, 1, 3, 4).reshape(B * T, C, H, W)
        qkv = F.conv2d(norm(f, f"{name}.norm"), w[f"{name}.to_qkv.weight"], w[f"{name}.to_qkv.bias"])
        seq = qkv.flatten(2).transpose(1, 2)                       # [BT, HW, 3C]
        q, k, v = seq.split(C, dim=-1)
        o = F.scaled_dot_product_attention(q.unsqueeze(1), k.unsqueeze(1), v.unsqueeze(1)).squeeze(1)
        o = o.transpose(1, 2).reshape(B * T, C, H, W)
        o = F.conv2d(o, w[f"{name}.proj.weight"], w[f"{name}.proj.bias"])
        return o.reshape(B, T, C, H, W).permute(0, 2, 1, 3, 4) + x

    def up2d(x, name):
        B, C, T, H, W = x.shape
        f = x.permute(0, 2, 1, 3, 4).reshape(B * T, C, H, W)
        f = F.interpolate(f, scale_factor=(2.0, 2.0), mode="nearest-exact")
        f = F.conv2d(f, w[f"{name}.weight"], w[f"{name}.bias"], padding=1)
        return f.reshape(B, T, -1, 2 * H, 2 * W).permute(0, 2, 1, 3, 4)

    x = F.conv3d(torch.from_numpy(np.asarray(z, dtype=np.float64)), w["post_quant_conv.weight"], w["post_quant_conv.bias"])
    x = cconv(x, "decoder.conv_in")
    x = resnet(x, "decoder.mid_block.resnets.0")
    x = attn(x, "decoder.mid_block.attentions.0")
    x = resnet(x, "decoder.mid_block.resnets.1")
    wan21 = w["post_quant_conv.weight"].shape[0] == 16
    specs = [(True, True), (True, True), (False, True), (False, False)]
    for i, (temporal, spatial) in enumerate(specs):
        name = f"decoder.up_blocks.{i}"
        ups = f"{name}.upsamplers.0" if wan21 else f"{name}.upsampler"
        inp = x
        for j in range(3):
            x = resnet(x, f"{name}.resnets.{j}")
        if not spatial:
            continue
        if temporal:
            B, C, T, H, W = x.shape
            y = cconv(x[:, :, 1:], f"{ups}.time_conv")                  # [B, 2C, T-1, H, W]
            y = y.reshape(B, 2, C, T - 1, H, W).permute(0, 2, 3, 1, 4, 5).reshape(B, C, 2 * (T - 1), H, W)
            x = torch.cat([x[:, :, :1], y], dim=2)
        x = up2d(x, f"{ups}.resample.1")
        if wan21:
            continue
        if temporal:   # r = 8: nearest x2 in t, h, w, the first frame kept once
            d = inp.repeat_interleave(2, 2).repeat_interleave(2, 3).repeat_interleave(2, 4)[:, :, 1:]
        else:          # r = 2: channel pair (2c, 2c+1) becomes row pair, each value in two columns
            B, C, T, H, W = inp.shape
            d = inp.reshape(B, C // 2, 2, T, H, W).permute(0, 1, 3, 4, 2, 5).reshape(B, C // 2, T, 2 * H, W)
            d = d.repeat_interleave(2, 4)
        x = x + d
    x = F.silu(norm(x, "decoder.norm_out"))
    out = cconv(x, "decoder.conv_out")                                   # [B, 12, F, h, w]
    if wan21:
        return out.numpy()
    B, _, Fr, H, W = out.shape
    # channel 4k + 2j + i -> colour k, row offset i, column offset j
    v = out.reshape(B, 3, 2, 2, Fr, H, W).permute(0, 1, 4, 5, 3, 6, 2).reshape(B, 3, Fr, 2 * H, 2 * W)
    return v.numpy()
