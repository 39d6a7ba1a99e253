"""Host-side checks of the C-ABI library that need no GPU: it loads, it exports
every entry point that include/tt.h declares, and argument errors that the host
catches before touching the device are reported with their status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tt():
    from block_diffusion_decoding_attn_b300 import build
    build.build()
    import block_diffusion_decoding_attn_b300 as tt
    return tt


def _declared():
    src = open(os.path.join(ROOT, "include", "tt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tt_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(tt):
    names = _declared()
    assert "tt_block_attn" in names and "tt_commit" in names
    lib = tt.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_host_argument_errors(tt):
    lib = tt.lib()
    assert lib.tt_status_string(-2) == b"TT_ERR_UNSUPPORTED"
    assert lib.tt_status_string(-4) == b"TT_ERR_TIMEOUT"
    assert lib.tt_status_string(-5) == b"TT_ERR_DEVICE_CHECK"
    # NULL handle is rejected before anything else
    rc = lib.tt_commit(None, None, 1, 1, 4, None, 1, None, None, None)
    assert rc == -1 and b"handle" in lib.tt_last_error()
    rc = lib.tt_commit_threshold(None, None, 1, 1, 4, None, 0.8, 1, None, None, None)
    assert rc == -1
    d = tt.AttnDesc(1, 8, 4, 1, 64, 16, 0.0)
    assert lib.tt_block_attn(None, ctypes.byref(d), *([None] * 7), None) == -1
    assert lib.tt_create(None, 0) == -1
    assert lib.tt_reserve(None, ctypes.byref(d), 1, 1) == -1
    assert lib.tt_set_attn_schedule(None, 0, 0, 0, 0) == -1
    assert lib.tt_commit_keys(None, None, None, 1, None) == -1
    assert lib.tt_get_error(None, None) == -1
    assert lib.tt_status_string(-6) == b"TT_ERR_NOT_READY"
    assert lib.tt_sync(None, None, 0, None) == -1 and b"tt_sync" in lib.tt_last_error()
    # the context-tower update and the training layout check the handle first too
    assert lib.tt_block_attn_causal(None, ctypes.byref(d), *([None] * 7), None) == -1
    assert lib.tt_kv_append(None, ctypes.byref(d), *([None] * 5), None) == -1
    assert b"tt_kv_append" in lib.tt_last_error()
    t = tt.TrainDesc(1, 64, 16, 4, 1, 64, 0.0)
    assert lib.tt_block_attn_train(None, ctypes.byref(t), *([None] * 6), None) == -1
    assert b"tt_block_attn_train" in lib.tt_last_error()
    # the LM head and the commit behind it
    assert lib.tt_lm_head(None, None, None, 1, 8, 4, None, None) == -1
    assert lib.tt_commit_rowmax(None, None, 1, 1, 4, None, 1, None, None, None) == -1
    assert lib.tt_block_attn_launches(None, ctypes.byref(d)) == -1
    # the allocation-free commit checks its size bound before touching a device
    assert lib.tt_commit_noalloc(None, 257, 256, 4, None, 1, None, None, None) == -2
    assert b"65536" in lib.tt_last_error()
    assert lib.tt_commit_noalloc(None, 1, 1, 4, None, 0, None, None, None) == -1


def test_status_codes_agree_with_the_header(tt):
    # every tt_status value of the header: the binding's constant of the same
    # name and the library's name for it
    src = open(os.path.join(ROOT, "include", "tt.h")).read()
    codes = dict((n, int(v)) for n, v in re.findall(r"\b(TT_(?:OK|ERR_[A-Z_]+))\s*=\s*(-?\d+)", src))
    assert codes["TT_OK"] == 0 and len(codes) >= 7
    for name, value in codes.items():
        assert getattr(tt, name) == value, name
        assert tt.lib().tt_status_string(value) == name.encode()
    bits = dict((n, int(v)) for n, v in re.findall(r"#define\s+(TT_DEV_[A-Z_]+)\s+(\d+)", src))
    assert bits and all(getattr(tt, n) == v for n, v in bits.items())


def test_create_without_gpu_fails_cleanly(tt):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = tt.lib().tt_create(ctypes.byref(h), 0)
    assert rc == -3 and not h.value
