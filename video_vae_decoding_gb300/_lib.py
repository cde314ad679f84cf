"""ctypes declarations of the C ABI in include/wan_vae.h (marshalling only)."""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libwanvae.so")

WAN_F32, WAN_BF16 = 0, 1

STATUS = {
    0: "WAN_OK", 1: "WAN_ERR_INVALID_ARG", 2: "WAN_ERR_DTYPE", 3: "WAN_ERR_MISSING_WEIGHT", 4: "WAN_ERR_SHAPE",
    5: "WAN_ERR_UNSUPPORTED", 6: "WAN_ERR_OOM", 7: "WAN_ERR_CUDA", 8: "WAN_ERR_STATE", 9: "WAN_ERR_INTERNAL",
    10: "WAN_ERR_NOT_IMPLEMENTED",
}


class WanTensor(ctypes.Structure):
    _fields_ = [
        ("name", ctypes.c_char_p),
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 5),
    ]


class WanProfile(ctypes.Structure):
    _fields_ = [
        ("launches", ctypes.c_int64),
        ("tc_launches", ctypes.c_int64),
        ("tc_ms", ctypes.c_double),
        ("tc_flops", ctypes.c_double),
        ("kind_ms", ctypes.c_double * 7),
        ("kind_work", ctypes.c_double * 7),
        ("kind_launches", ctypes.c_int64 * 7),
        ("tc_exec_flops", ctypes.c_double),
        ("kind_exec", ctypes.c_double * 7),
    ]


PROFILE_KINDS = ("conv3x3x3", "time_conv", "upsample2d_conv", "attention_gemm", "conv_out", "rms_norm", "misc_memory")
PROFILE_TENSOR_KINDS = 5  # the first five report FLOPs, the rest bytes

_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64

# name -> (restype, argtypes)
SIGNATURES = {
    "wan_vae_out_frames": (_i64, [_i64]),
    "wan_vae_last_error": (ctypes.c_char_p, []),
    "wan_vae_status_string": (ctypes.c_char_p, [_i32]),
    "wan_vae_model_create": (_i32, [ctypes.POINTER(WanTensor), _i32, _i32, _vp, ctypes.POINTER(_vp)]),
    "wan_vae_model_destroy": (None, [_vp]),
    "wan_vae_model_base_dim": (_i32, [_vp]),
    "wan_vae_model_z_dim": (_i32, [_vp]),
    "wan_vae_model_scale": (_i32, [_vp]),
    "wan_vae_model_set_latent_stats": (_i32, [_vp, _vp, _vp, _i32]),
    "wan_vae_stream_create": (_i32, [_vp, _i32, _i32, _i32, _i32, ctypes.POINTER(_vp)]),
    "wan_vae_stream_reset": (_i32, [_vp, _vp]),
    "wan_vae_stream_destroy": (None, [_vp]),
    "wan_vae_stream_workspace_bytes": (_i64, [_vp]),
    "wan_vae_stream_sync_status": (_i32, [_vp, _vp]),
    "wan_vae_stream_state_bytes": (_i64, [_vp]),
    "wan_vae_stream_save": (_i32, [_vp, _vp, _i64, _vp]),
    "wan_vae_stream_load": (_i32, [_vp, _vp, _i64, _vp]),
    "wan_vae_stream_profile_begin": (_i32, [_vp]),
    "wan_vae_stream_profile_end": (_i32, [_vp, _vp, ctypes.POINTER(WanProfile)]),
    "wan_vae_decode_chunk": (_i32, [_vp, _vp, _i32, _i64, _i64, _i32, _vp, _i32, _i64, _i64, _vp, _vp]),
    "wan_vae_decode_clip": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _vp, _vp]),
    "wan_vae_decode_clip_host": (_i32, [_vp, _vp, _i32, _i32, _vp, _i32, _vp]),
    "wan_vae_decode": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(WanTensor), _i32, _vp, _i32, _vp]),
    "wan_vae_decode_tiled": (_i32, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                    _vp, _i32, _vp]),
    "wan_attention_block": (_i32, [_vp, _i32, _i32, _i32, _i32, ctypes.POINTER(WanTensor), _i32, _vp, _vp]),
    "wan_attention_create": (_i32, [ctypes.POINTER(WanTensor), _i32, _i32, _i32, _i32, _i32, _vp,
                                    ctypes.POINTER(_vp)]),
    "wan_attention_run": (_i32, [_vp, _vp, _vp, _vp]),
    "wan_attention_status": (_i32, [_vp, _vp]),
    "wan_attention_destroy": (None, [_vp]),
    "wan_causal_conv3d": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                 _vp, _vp]),
    "wan_conv_out_video": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _i32, _vp,
                                  _vp]),
    "wan_selftest_wait_timeout": (_i32, [_i32, ctypes.POINTER(_i32), _vp]),
    "wan_selftest_attention_timeout": (_i32, [_i32, ctypes.POINTER(_i32), _vp]),
    "wan_causal_conv3d_noalloc": (_i32, [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _i32,
                                         _i32, _vp, _vp]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libwanvae.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m video_vae_decoding_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class WanError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def check(status: int) -> None:
    if status != 0:
        msg = load().wan_vae_last_error()
        raise WanError(status, msg.decode() if msg else "")
