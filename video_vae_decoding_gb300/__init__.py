"""GB300 (sm_103a) Wan VAE decode: the Wan2.2-TI2V-5B decoder, and the Wan2.1
decoder when given its weights.

A thin Python binding over the C ABI of ``include/wan_vae.h``: it only
marshals torch CUDA tensors (device memory, streams) into the library's
calls.  Every step of the decode runs in the library's CUDA kernels; if the
library is not built, calls raise instead of falling back to anything else.

Typical use::

    model = Model(weights, dtype=torch.bfloat16)   # packs the decoder once
    stream = DecodeStream(model, B, h, w)           # causal caches + workspace
    video = stream.decode_clip(z)                   # [B, 3, 4T-3, 16h, 16w]
    stream.decode_chunk(z, t0, n, out, out_f0)      # or chunk by chunk
    tiled = model.decode_tiled(z, tile=(256, 256), stride=(192, 192))
    model.set_latent_stats(mean, std)               # de-normalise latents first

``decode(z, weights, dtype)`` is the one-shot form.
"""

from __future__ import annotations

import ctypes

import torch

from ._lib import PROFILE_KINDS, WAN_BF16, WAN_F32, WanError, WanProfile, WanTensor, check, load  # noqa: F401

__all__ = ["Model", "DecodeStream", "decode", "attention_block", "causal_conv3d", "out_frames", "WanError"]


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return WAN_F32
    if dtype == torch.bfloat16:
        return WAN_BF16
    raise ValueError(f"dtype must be torch.float32 or torch.bfloat16, not {dtype}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def out_frames(T: int) -> int:
    return int(load().wan_vae_out_frames(T))


def weight_table(weights: "dict[str, torch.Tensor]"):
    """wan_tensor array describing `weights` (kept alive by the returned list)."""
    items = list(weights.items())
    arr = (WanTensor * len(items))()
    keep = []
    for i, (name, t) in enumerate(items):
        if t.dim() > 5:
            raise ValueError(f"{name}: more than 5 dimensions")
        bname = name.encode()
        keep.append(bname)
        keep.append(t)
        arr[i].name = bname
        arr[i].data = _dev(t, name)
        arr[i].dtype = {torch.float32: WAN_F32, torch.bfloat16: WAN_BF16}.get(t.dtype, 99)
        arr[i].ndim = t.dim()
        for d in range(t.dim()):
            arr[i].shape[d] = t.shape[d]
    return arr, keep


class Model:
    """Packed decoder weights (wan_vae_model_create)."""

    def __init__(self, weights: "dict[str, torch.Tensor]", dtype: torch.dtype = torch.bfloat16, stream=None):
        lib = load()
        arr, keep = weight_table(weights)
        h = ctypes.c_void_p()
        check(lib.wan_vae_model_create(arr, len(keep) // 2, _code(dtype), _stream(stream), ctypes.byref(h)))
        self._h = h
        self.dtype = dtype

    @property
    def handle(self):
        return self._h

    @property
    def base_dim(self) -> int:
        return int(load().wan_vae_model_base_dim(self._h))

    @property
    def z_dim(self) -> int:
        """Latent channels: 48 (TI2V-5B) or 16 (Wan2.1)."""
        return int(load().wan_vae_model_z_dim(self._h))

    @property
    def scale(self) -> int:
        """Video pixels per latent along h and w: 16 (TI2V-5B) or 8 (Wan2.1)."""
        return int(load().wan_vae_model_scale(self._h))

    def set_latent_stats(self, mean=None, std=None):
        """Latent de-normalisation (wan_vae_model_set_latent_stats): later decodes
        through this model map z to z * std + mean per latent channel first.
        mean, std: z_dim values each (sequence, array or tensor); both None: off."""
        if mean is None and std is None:
            check(load().wan_vae_model_set_latent_stats(self._h, None, None, 0))
            return
        m = torch.as_tensor(mean, dtype=torch.float32).detach().cpu().contiguous().reshape(-1)
        s = torch.as_tensor(std, dtype=torch.float32).detach().cpu().contiguous().reshape(-1)
        if m.numel() != s.numel():
            raise ValueError(f"{m.numel()} means but {s.numel()} stds")
        check(load().wan_vae_model_set_latent_stats(self._h, m.data_ptr(), s.data_ptr(), m.numel()))

    def decode_tiled(self, z: torch.Tensor, tile=(256, 256), stride=(192, 192), out_dtype: torch.dtype = None,
                     tile_batch: int = 0, max_chunk: int = 4, stream=None) -> torch.Tensor:
        """Tiled decode (wan_vae_decode_tiled): z [B, z_dim, T, h, w] on the GPU ->
        video [B, 3, 4T-3, scale*h, scale*w]; tile and stride are (height,
        width) in video pixels, multiples of `scale`."""
        B, _, T, h, w = z.shape
        dt = self.dtype if out_dtype is None else out_dtype
        k = self.scale
        out = torch.empty((B, 3, 4 * T - 3, k * h, k * w), device=z.device, dtype=dt)
        check(load().wan_vae_decode_tiled(self._h, _dev(z, "z"), _code(z.dtype), B, T, h, w, tile[0], tile[1],
                                          stride[0], stride[1], tile_batch, max_chunk, _dev(out, "out"), _code(dt),
                                          _stream(stream)))
        return out

    def close(self):
        if self._h:
            load().wan_vae_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecodeStream:
    """Causal caches + workspace for B x h x w latents (wan_vae_stream_create)."""

    def __init__(self, model: Model, B: int, h: int, w: int, max_chunk: int = 4):
        lib = load()
        s = ctypes.c_void_p()
        check(lib.wan_vae_stream_create(model.handle, B, h, w, max_chunk, ctypes.byref(s)))
        self._s = s
        self.model = model
        self.B, self.h, self.w, self.max_chunk = B, h, w, max_chunk

    @property
    def workspace_bytes(self) -> int:
        return int(load().wan_vae_stream_workspace_bytes(self._s))

    def reset(self, stream=None):
        check(load().wan_vae_stream_reset(self._s, _stream(stream)))

    def sync_status(self, stream=None):
        check(load().wan_vae_stream_sync_status(self._s, _stream(stream)))

    @property
    def state_bytes(self) -> int:
        return int(load().wan_vae_stream_state_bytes(self._s))

    def save_state(self, stream=None) -> torch.Tensor:
        """The causal caches and chunk position, as a uint8 device tensor."""
        buf = torch.empty(self.state_bytes, dtype=torch.uint8, device="cuda")
        check(load().wan_vae_stream_save(self._s, buf.data_ptr(), buf.numel(), _stream(stream)))
        return buf

    def load_state(self, buf: torch.Tensor, stream=None):
        if not buf.is_contiguous():
            raise ValueError("state buffer must be contiguous")
        check(load().wan_vae_stream_load(self._s, buf.data_ptr(), buf.numel(), _stream(stream)))

    def profile_begin(self):
        check(load().wan_vae_stream_profile_begin(self._s))

    def profile_end(self, stream=None) -> dict:
        """Waits for the stream; returns launch counts and the summed device
        time and nominal FLOPs of the tensor-core launches since profile_begin."""
        p = WanProfile()
        check(load().wan_vae_stream_profile_end(self._s, _stream(stream), ctypes.byref(p)))
        kinds = {}
        for i, k in enumerate(PROFILE_KINDS):
            row = {"ms": p.kind_ms[i], "launches": p.kind_launches[i]}
            if i < 5:
                row["flops"], row["exec_flops"] = p.kind_work[i], p.kind_exec[i]
            else:
                row["bytes"] = p.kind_work[i]
            kinds[k] = row
        return {"launches": p.launches, "tc_launches": p.tc_launches, "tc_ms": p.tc_ms, "tc_flops": p.tc_flops,
                "tc_exec_flops": p.tc_exec_flops, "kinds": kinds}

    def decode_chunk(self, z, t0, n, out, out_f0, preclamp=None, stream=None):
        p = 0 if preclamp is None else _dev(preclamp, "preclamp")
        check(load().wan_vae_decode_chunk(self._s, _dev(z, "z"), _code(z.dtype), z.shape[2], t0, n, _dev(out, "out"),
                                          _code(out.dtype), out.shape[2], out_f0, p or None, _stream(stream)))

    def decode_clip(self, z, out=None, out_dtype=None, preclamp=None, stream=None):
        B, _, T, h, w = z.shape
        if out is None:
            k = self.model.scale
            out = torch.empty((B, 3, 4 * T - 3, k * h, k * w), device=z.device,
                              dtype=out_dtype or self.model.dtype)
        p = 0 if preclamp is None else _dev(preclamp, "preclamp")
        check(load().wan_vae_decode_clip(self._s, _dev(z, "z"), _code(z.dtype), T, _dev(out, "out"), _code(out.dtype),
                                         p or None, _stream(stream)))
        return out

    def decode_clip_host(self, z_host: torch.Tensor, out_host: torch.Tensor, stream=None):
        """z_host, out_host: CPU tensors (pinned recommended); blocks until done."""
        for t, n in ((z_host, "z_host"), (out_host, "out_host")):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{n} must be a contiguous host tensor")
        check(load().wan_vae_decode_clip_host(self._s, z_host.data_ptr(), _code(z_host.dtype), z_host.shape[2],
                                              out_host.data_ptr(), _code(out_host.dtype), _stream(stream)))
        return out_host

    def close(self):
        if self._s:
            load().wan_vae_stream_destroy(self._s)
            self._s = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode(z: torch.Tensor, weights: "dict[str, torch.Tensor]", dtype: torch.dtype = torch.float32, stream=None):
    """One-shot decode(z, weights, dtype) -> video [B, 3, 4T-3, 16h, 16w] of `dtype`
    (Wan2.1 weights, z [B, 16, T, h, w]: [B, 3, 4T-3, 8h, 8w])."""
    code = _code(dtype)
    B, C, T, h, w = z.shape
    k = 8 if C == 16 else 16
    out = torch.empty((B, 3, 4 * T - 3, k * h, k * w), device=z.device, dtype=dtype)
    arr, keep = weight_table(weights)
    check(load().wan_vae_decode(_dev(z, "z"), _code(z.dtype), B, T, h, w, arr, len(keep) // 2, _dev(out, "out"), code,
                                _stream(stream)))
    return out


def attention_block(x: torch.Tensor, weights: "dict[str, torch.Tensor]", H: int, W: int, stream=None):
    """x [N, H*W, C] bf16 channels-last -> attention(x) + x, same layout."""
    N, HW, C = x.shape
    out = torch.empty_like(x)
    arr, keep = weight_table(weights)
    check(load().wan_attention_block(_dev(x, "x"), N, H, W, C, arr, len(keep) // 2, _dev(out, "out"),
                                     _stream(stream)))
    return out


class AttentionBlock:
    """The mid-block attention with its weights packed once
    (wan_attention_create / _run / _destroy) for N frames of H x W positions."""

    def __init__(self, weights: "dict[str, torch.Tensor]", N: int, H: int, W: int, C: int, stream=None):
        arr, keep = weight_table(weights)
        h = ctypes.c_void_p()
        check(load().wan_attention_create(arr, len(keep) // 2, N, H, W, C, _stream(stream), ctypes.byref(h)))
        self._h = h
        self.N, self.H, self.W, self.C = N, H, W, C

    def __call__(self, x: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
        if tuple(x.shape) != (self.N, self.H * self.W, self.C) or x.dtype != torch.bfloat16:
            raise ValueError(f"x must be bf16 [{self.N}, {self.H * self.W}, {self.C}]")
        out = torch.empty_like(x) if out is None else out
        check(load().wan_attention_run(self._h, _dev(x, "x"), _dev(out, "out"), _stream(stream)))
        return out

    def sync_status(self, stream=None):
        """Waits for the stream; raises if a run recorded a bounded-wait timeout."""
        check(load().wan_attention_status(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            load().wan_attention_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


def conv_out_video(x: torch.Tensor, n_hist: int, weight: torch.Tensor, bias: torch.Tensor, out_dtype=torch.bfloat16,
                   preclamp: bool = False, stream=None):
    """x [B, n_hist + F, H, W, Cin] bf16 channels-last -> the clamped video
    [B, 3, F, 2H, 2W] (weight [12, Cin, 3, 3, 3]) or [B, 3, F, H, W] (weight
    [3, Cin, 3, 3, 3]); with preclamp, also the fp32 values before the clamp."""
    B, Ft, H, W, Cin = x.shape
    Cout = weight.shape[0]
    F = Ft - n_hist
    p = 2 if Cout == 12 else 1
    out = torch.empty((B, 3, F, p * H, p * W), device=x.device, dtype=out_dtype)
    pre = torch.empty(out.shape, device=x.device, dtype=torch.float32) if preclamp else None
    if weight.dtype != bias.dtype:
        raise ValueError("weight and bias must share a dtype")
    check(load().wan_conv_out_video(_dev(x, "x"), B, n_hist, F, H, W, Cin, _dev(weight, "weight"), _dev(bias, "bias"),
                                    _code(weight.dtype), Cout, _dev(out, "out"), _code(out_dtype),
                                    _dev(pre, "preclamp") if pre is not None else None, _stream(stream)))
    return (out, pre) if preclamp else out


def causal_conv3d(x: torch.Tensor, n_hist: int, weight: torch.Tensor, bias: torch.Tensor, stream=None):
    """x [B, n_hist + F, H, W, Cin] bf16 channels-last -> [B, F, H, W, Cout] bf16."""
    B, Ft, H, W, Cin = x.shape
    Cout, _, kt, kh, kw = weight.shape
    F = Ft - n_hist
    out = torch.empty((B, F, H, W, Cout), device=x.device, dtype=torch.bfloat16)
    if weight.dtype != bias.dtype:
        raise ValueError("weight and bias must share a dtype")
    check(load().wan_causal_conv3d(_dev(x, "x"), B, n_hist, F, H, W, Cin, _dev(weight, "weight"), _dev(bias, "bias"),
                                   _code(weight.dtype), Cout, kt, kh, kw, _dev(out, "out"), _stream(stream)))
    return out
