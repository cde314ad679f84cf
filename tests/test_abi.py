"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments on the host (no GPU needed: these calls return before
any CUDA work)."""

import ctypes
import os
import re

import pytest

import wan_synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from video_vae_decoding_gb300 import build
    build.build()
    from video_vae_decoding_gb300 import _lib
    return _lib.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "wan_vae.h")).read()
    return sorted(set(re.findall(r"^\s*(?:wan_status|void|int64_t|int32_t|const char\*)\s+(wan_\w+)\s*\(", text, re.M)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_binding_declares_every_header_function():
    # the ctypes table gives every declared entry point its argument and
    # return types (an entry point without one would be called untyped)
    from video_vae_decoding_gb300._lib import SIGNATURES
    missing = [n for n in _declared() if n not in SIGNATURES]
    assert not missing, missing


def test_out_frames(lib):
    assert [lib.wan_vae_out_frames(t) for t in (0, 1, 2, 31, 21)] == [0, 1, 5, 121, 81]


def test_status_strings(lib):
    assert lib.wan_vae_status_string(0) == b"WAN_OK"
    assert lib.wan_vae_status_string(2) == b"WAN_ERR_DTYPE"


def _table(base=16, drop=None, reshape=None, dtype=0):
    from video_vae_decoding_gb300._lib import WanTensor
    shapes = wan_synth.weight_shapes(base)
    items = [(k, v) for k, v in shapes.items() if k != drop]
    arr = (WanTensor * (len(items) + 1))()
    keep = []
    for i, (k, shp) in enumerate(items):
        if reshape and k == reshape[0]:
            shp = reshape[1]
        nm = k.encode()
        keep.append(nm)
        arr[i].name = nm
        arr[i].data = 0x1000 + 256 * i      # never dereferenced: validation fails or stops first
        arr[i].dtype = dtype
        arr[i].ndim = len(shp)
        for d, x in enumerate(shp):
            arr[i].shape[d] = x
    # a foreign name is ignored
    arr[len(items)].name = b"encoder.conv_in.weight"
    arr[len(items)].data = 0x10
    arr[len(items)].dtype = 0
    arr[len(items)].ndim = 1
    arr[len(items)].shape[0] = 3
    return arr, len(items) + 1, keep


def _create(lib, table, n, dtype):
    h = ctypes.c_void_p()
    return lib.wan_vae_model_create(table, n, dtype, None, ctypes.byref(h)), h


def test_model_create_validation(lib):
    arr, n, keep = _table()
    assert _create(lib, arr, n, 7)[0] == 2                        # WAN_ERR_DTYPE (the page's ValueError)
    arr, n, keep = _table(drop="decoder.up_blocks.2.resnets.0.conv_shortcut.bias")
    st, _ = _create(lib, arr, n, 1)
    assert st == 3 and b"conv_shortcut.bias" in lib.wan_vae_last_error()
    arr, n, keep = _table(reshape=("decoder.up_blocks.1.upsampler.time_conv.weight", (128, 64, 3, 3, 3)))
    st, _ = _create(lib, arr, n, 1)
    assert st == 4 and b"time_conv" in lib.wan_vae_last_error()
    arr, n, keep = _table(reshape=("decoder.norm_out.gamma", (15,)))
    assert _create(lib, arr, n, 1)[0] == 4
    arr, n, keep = _table(dtype=5)
    assert _create(lib, arr, n, 1)[0] == 2
    assert lib.wan_vae_model_create(arr, n, 1, None, None) == 1


def test_call_validation_without_device(lib):
    vp = ctypes.c_void_p
    assert lib.wan_vae_decode_chunk(None, vp(1), 1, 1, 0, 1, vp(1), 1, 1, 0, None, None) == 1
    assert lib.wan_vae_decode_clip(None, vp(1), 1, 1, vp(1), 1, None, None) == 1
    assert lib.wan_vae_decode(vp(1), 1, 1, 1, 4, 4, None, 0, vp(1), 9, None) == 2
    assert lib.wan_vae_decode(vp(1), 3, 1, 1, 4, 4, None, 0, vp(1), 1, None) == 2
    assert lib.wan_vae_stream_create(None, 1, 4, 4, 1, ctypes.byref(vp())) == 1
    assert lib.wan_causal_conv3d(vp(1), 1, 0, 1, 4, 4, 64, vp(1), vp(1), 0, 64, 3, 2, 3, vp(1), None) == 5
    assert lib.wan_causal_conv3d(vp(1), 1, 3, 1, 4, 4, 64, vp(1), vp(1), 0, 64, 3, 3, 3, vp(1), None) == 1
    assert lib.wan_attention_block(vp(1), 1, 4, 4, 48, None, 0, vp(1), None) == 1
    f48 = (ctypes.c_float * 48)()
    assert lib.wan_vae_model_set_latent_stats(None, f48, f48, 48) == 1
    # tiled decode: tile arguments are checked before anything else
    tiled = lambda th, tw, sh, sw, tb=0, mc=4, zd=1, od=1: lib.wan_vae_decode_tiled(  # noqa: E731
        None, vp(16), zd, 1, 1, 4, 4, th, tw, sh, sw, tb, mc, vp(16), od, None)
    assert tiled(250, 256, 192, 192) == 1           # not a multiple of 16
    assert tiled(256, 256, 256, 272) == 1           # stride larger than the tile
    assert tiled(256, 256, 0, 192) == 1
    assert tiled(256, 256, 192, 192, tb=-1) == 1
    assert tiled(256, 256, 192, 192, mc=0) == 1
    assert tiled(256, 256, 192, 192, zd=7) == 2
    assert tiled(256, 256, 192, 192) == 1           # null model
    assert b"model" in lib.wan_vae_last_error()
    from video_vae_decoding_gb300._lib import WanTensor
    assert lib.wan_attention_block(vp(1), 1, 4, 4, 48, (WanTensor * 1)(), 0, vp(1), None) == 5


def test_binding_rejects_bad_dtype():
    import torch
    import video_vae_decoding_gb300 as wv
    with pytest.raises(ValueError):
        wv._code(torch.float16)
