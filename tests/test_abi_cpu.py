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
    assert lib.tt_commit_workspace_bytes(4, 32) == 1024 + 512 + 16
    assert lib.tt_commit_workspace_bytes(-1, 3) == 0
    assert lib.tt_status_string(-2) == b"TT_ERR_UNSUPPORTED"
    # NULL handle is rejected before anything else
    rc = lib.tt_commit(None, None, 1, 1, 4, None, 1, None, None, None, 0, None)
    assert rc == -1 and b"handle" in lib.tt_last_error()
    d = tt.AttnDesc(1, 8, 4, 1, 64, 16, 0.0, 0)
    assert lib.tt_block_attn(None, ctypes.byref(d), *([None] * 7), None, 0, None) == -1
    assert lib.tt_block_attn_workspace_bytes(None, ctypes.byref(d)) == 0
    assert lib.tt_create(None, 0) == -1
    # the context-tower update and the training layout check the handle first too
    assert lib.tt_block_attn_causal(None, ctypes.byref(d), *([None] * 7), None, 0, None) == -1
    assert lib.tt_kv_append(None, ctypes.byref(d), *([None] * 5), None) == -1
    assert b"tt_kv_append" in lib.tt_last_error()
    t = tt.TrainDesc(1, 64, 16, 4, 1, 64, 0.0, 0)
    assert lib.tt_block_attn_train(None, ctypes.byref(t), *([None] * 6), None, 0, None) == -1
    assert b"tt_block_attn_train" in lib.tt_last_error()
    assert lib.tt_block_attn_train_workspace_bytes(None, ctypes.byref(t)) == 0


def test_create_without_gpu_fails_cleanly(tt):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = tt.lib().tt_create(ctypes.byref(h), 0)
    assert rc == -3 and not h.value
