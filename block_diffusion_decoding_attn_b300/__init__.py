"""TwoTower denoising-step hot path on B300 (sm_103a): block attention and
unmask/commit, as hand-written CUDA kernels behind the C ABI in ``include/tt.h``.

This module is argument marshalling only: it turns torch tensors (device
memory, streams) into the plain pointers and sizes of the C ABI and calls
``libtt.so``. Every step of the computation runs in the library's kernels.
There is no CPU fallback: without the built library or a CUDA device every
entry point raises.

Entry points mirror the C ABI:

* :func:`block_attn` -> ``tt_block_attn`` ("Nemotron-Labs-TwoTower",
  Section 2.1, Eq. 1)
* :func:`commit` -> ``tt_commit`` (Section 2.2, Algorithm 2 with k commits per
  block per step)
* :func:`commit_threshold` -> ``tt_commit_threshold`` (Algorithm 2 with a
  confidence threshold gamma and a floor of ceil(#masked / steps_left))
* :func:`block_attn_train` -> ``tt_block_attn_train`` (Section 2.3: all noisy
  blocks of a clean sequence in one pass)
* :func:`block_attn` with ``causal=True`` -> ``tt_block_attn_causal`` and
  :func:`kv_append` -> ``tt_kv_append``: the context tower's update after a
  commit (Section 2.1, Algorithm 1)
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtt.so")

TT_OK = 0
TT_ERR_INVALID_ARG, TT_ERR_UNSUPPORTED, TT_ERR_CUDA, TT_ERR_TIMEOUT, TT_ERR_DEVICE_CHECK = (
    -1, -2, -3, -4, -5)
TT_ERR_NOT_READY = -6
TT_DEV_CTX_LEN_RANGE = 1
TT_DEV_WAIT_TIMEOUT = 2

_lock = threading.Lock()
_lib = None
_handles: dict[int, "Handle"] = {}


class TTError(RuntimeError):
    """A C-ABI call returned an error status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Loads libtt.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: run block_diffusion_decoding_attn_b300."
                                  "build.build() (nvcc, sm_103a) first")
            L = ctypes.CDLL(LIB_PATH)
            P, I = ctypes.c_void_p, ctypes.c_int
            L.tt_create.argtypes = [ctypes.POINTER(P), I]
            L.tt_destroy.argtypes = [P]
            L.tt_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
            L.tt_sync.argtypes = [P, P, ctypes.c_uint, ctypes.POINTER(ctypes.c_int)]
            L.tt_set_wait_timeout.argtypes = [P, ctypes.c_ulonglong]
            L.tt_set_attn_schedule.argtypes = [P, I, I, I, I]
            L.tt_reserve.argtypes = [P, ctypes.POINTER(AttnDesc), I, I]
            L.tt_status_string.restype = ctypes.c_char_p
            L.tt_status_string.argtypes = [I]
            L.tt_last_error.restype = ctypes.c_char_p
            L.tt_last_error.argtypes = []
            L.tt_block_attn_launches.argtypes = [P, ctypes.POINTER(AttnDesc)]
            L.tt_block_attn.argtypes = [P, ctypes.POINTER(AttnDesc)] + [P] * 7 + [P]
            L.tt_block_attn_causal.argtypes = L.tt_block_attn.argtypes
            L.tt_kv_append.argtypes = [P, ctypes.POINTER(AttnDesc)] + [P] * 5 + [P]
            L.tt_block_attn_train.argtypes = [P, ctypes.POINTER(TrainDesc)] + [P] * 6 + [P]
            L.tt_commit.argtypes = [P, P, I, I, I, P, I, P, P, P]
            L.tt_commit_threshold.argtypes = [P, P, I, I, I, P, ctypes.c_double, I, P, P, P]
            L.tt_commit_keys.argtypes = [P, P, P, I, P]
            L.tt_commit_noalloc.argtypes = [P, I, I, I, P, I, P, P, P]
            L.tt_lm_head.argtypes = [P, P, P, I, I, I, P, P]
            L.tt_commit_rowmax.argtypes = [P, P, I, I, I, P, I, P, P, P]
            L.tt_commit_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
            for f in ("tt_create", "tt_destroy", "tt_get_error", "tt_set_wait_timeout",
                      "tt_set_attn_schedule", "tt_reserve", "tt_block_attn", "tt_block_attn_launches",
                      "tt_block_attn_causal", "tt_kv_append", "tt_block_attn_train", "tt_commit",
                      "tt_commit_threshold", "tt_commit_keys", "tt_commit_noalloc",
                      "tt_commit_noalloc_status", "tt_lm_head", "tt_commit_rowmax"):
                getattr(L, f).restype = I
            _lib = L
    return _lib


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("ctx_cap", ctypes.c_int),
                ("scale", ctypes.c_float)]


class TrainDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("N", ctypes.c_int), ("S", ctypes.c_int),
                ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("scale", ctypes.c_float)]


def _check(status: int, what: str):
    if status != TT_OK:
        L = lib()
        msg = L.tt_last_error().decode() or L.tt_status_string(status).decode()
        raise TTError(status, f"{what}: {msg}")


class Handle:
    """A library handle bound to one CUDA device (``tt_create``)."""

    def __init__(self, device: int = 0):
        self.device = device
        self._h = ctypes.c_void_p()
        _check(lib().tt_create(ctypes.byref(self._h), device), "tt_create")

    @property
    def ptr(self):
        return self._h

    def get_error(self) -> int:
        """Synchronizes the device; returns and clears the TT_DEV_* status bits."""
        st = ctypes.c_int(0)
        rc = lib().tt_get_error(self._h, ctypes.byref(st))
        if rc not in (TT_OK, TT_ERR_TIMEOUT, TT_ERR_DEVICE_CHECK):
            _check(rc, "tt_get_error")
        return st.value

    def sync(self, stream=None, timeout_ms: int = 1000):
        """Waits on the host for at most timeout_ms for the work issued on
        `stream` (default: the current torch stream of the handle's device) to
        finish (tt_sync). Returns (done, status): done False if it was still
        running; status = the TT_DEV_* bits, not cleared."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        st = ctypes.c_int(0)
        rc = lib().tt_sync(self._h, ctypes.c_void_p(stream.cuda_stream), int(timeout_ms),
                           ctypes.byref(st))
        if rc == TT_ERR_NOT_READY:
            return False, 0
        _check(rc, "tt_sync")
        return True, st.value

    def set_wait_timeout(self, ns: int):
        _check(lib().tt_set_wait_timeout(self._h, int(ns)), "tt_set_wait_timeout")

    def set_attn_schedule(self, kernel: int = 0, max_ctas: int = 0, min_tiles: int = 0,
                          splits: int = 0):
        """Attention schedule (tt_set_attn_schedule): kernel 0 by shape, 1 one
        unit per CTA, 2 persistent; max_ctas / min_tiles for the persistent
        schedule; splits for the one-unit-per-CTA schedule (0 = defaults)."""
        _check(lib().tt_set_attn_schedule(self._h, int(kernel), int(max_ctas), int(min_tiles),
                                          int(splits)), "tt_set_attn_schedule")

    def reserve(self, attn: "AttnDesc | None" = None, commit_B: int = 0, commit_L: int = 0):
        """Grows the handle's scratch for these shapes now (so calls do not allocate)."""
        _check(lib().tt_reserve(self._h, ctypes.byref(attn) if attn is not None else None,
                                int(commit_B), int(commit_L)), "tt_reserve")

    def close(self):
        if self._h:
            lib().tt_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def handle(device: int | None = None) -> Handle:
    """The process-wide handle of `device` (default: torch's current device)."""
    import torch
    if device is None:
        device = torch.cuda.current_device()
    with _lock:
        h = _handles.get(device)
    if h is None:
        h = Handle(device)
        with _lock:
            _handles.setdefault(device, h)
            h = _handles[device]
    return h


def _stream_ptr(t, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def attn_desc(q, k_ctx, scale: float = 0.0) -> AttnDesc:
    B, L, Hq, D = q.shape
    Hkv, C = k_ctx.shape[1], k_ctx.shape[2]
    return AttnDesc(B, L, Hq, Hkv, D, C, float(scale))


def block_attn_launches(desc: AttnDesc, h: Handle | None = None) -> int:
    """Kernel launches one attention call with this descriptor makes (1 or 2)."""
    h = h or handle()
    n = int(lib().tt_block_attn_launches(h.ptr, ctypes.byref(desc)))
    if n < 0:
        _check(n, "tt_block_attn_launches")
    return n


def block_attn(q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, out=None, scale: float = 0.0,
               h: Handle | None = None, stream=None, causal: bool = False):
    """Block attention, Eq. (1): one softmax per query over [context keys; block keys].

    q [B][L][Hq][D], k_blk/v_blk [B][L][Hkv][D], k_ctx/v_ctx [B][Hkv][C_cap][D]
    (torch.bfloat16, CUDA, contiguous); ctx_len [B] int32 on the device.
    ``causal``: block query l sees block keys 0..l only (tt_block_attn_causal).
    Returns out [B][L][Hq][D] bf16.
    """
    import torch
    for name, t in (("q", q), ("k_blk", k_blk), ("v_blk", v_blk), ("k_ctx", k_ctx),
                    ("v_ctx", v_ctx)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if ctx_len.dtype != torch.int32 or not ctx_len.is_cuda:
        raise ValueError("ctx_len must be an int32 CUDA tensor")
    h = h or handle(q.device.index)
    desc = attn_desc(q, k_ctx, scale)
    if out is None:
        out = torch.empty_like(q)
    fn = lib().tt_block_attn_causal if causal else lib().tt_block_attn
    _check(fn(h.ptr, ctypes.byref(desc), _dev_ptr(q), _dev_ptr(k_blk), _dev_ptr(v_blk),
              _dev_ptr(k_ctx), _dev_ptr(v_ctx), _dev_ptr(ctx_len), _dev_ptr(out),
              _stream_ptr(q, stream)), "tt_block_attn_causal" if causal else "tt_block_attn")
    return out


def block_attn_train(q, k_noisy, v_noisy, k_clean, v_clean, S: int, out=None,
                     scale: float = 0.0, h: Handle | None = None, stream=None):
    """Training-time batched block attention (Section 2.3): noisy block j of each
    sequence attends to the clean keys of positions 0..j*S-1 and to its own S
    noisy keys.

    q [B][N][Hq][D], k_noisy/v_noisy [B][N][Hkv][D], k_clean/v_clean [B][Hkv][N][D]
    (torch.bfloat16, CUDA, contiguous), N a multiple of S. Returns out
    [B][N][Hq][D] bf16.
    """
    import torch
    for name, t in (("q", q), ("k_noisy", k_noisy), ("v_noisy", v_noisy), ("k_clean", k_clean),
                    ("v_clean", v_clean)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    B, N, Hq, D = q.shape
    Hkv = k_noisy.shape[2]
    if tuple(k_noisy.shape) != (B, N, Hkv, D) or tuple(v_noisy.shape) != (B, N, Hkv, D) or \
            tuple(k_clean.shape) != (B, Hkv, N, D) or tuple(v_clean.shape) != (B, Hkv, N, D):
        raise ValueError("block_attn_train: inconsistent shapes")
    h = h or handle(q.device.index)
    desc = TrainDesc(B, N, int(S), Hq, Hkv, D, float(scale))
    if out is None:
        out = torch.empty_like(q)
    _check(lib().tt_block_attn_train(h.ptr, ctypes.byref(desc), _dev_ptr(q), _dev_ptr(k_noisy),
                                     _dev_ptr(v_noisy), _dev_ptr(k_clean), _dev_ptr(v_clean),
                                     _dev_ptr(out), _stream_ptr(q, stream)),
           "tt_block_attn_train")
    return out


def kv_append(k_blk, v_blk, k_ctx, v_ctx, ctx_len, h: Handle | None = None, stream=None):
    """Appends the block's K/V to the cache in place and advances ctx_len by L.

    k_blk/v_blk [B][L][Hkv][D], k_ctx/v_ctx [B][Hkv][C_cap][D] (torch.bfloat16,
    CUDA, contiguous); ctx_len [B] int32 on the device, updated in place. A
    block that does not fit is skipped and flags TT_DEV_CTX_LEN_RANGE
    (Handle.get_error).
    """
    import torch
    for name, t in (("k_blk", k_blk), ("v_blk", v_blk), ("k_ctx", k_ctx), ("v_ctx", v_ctx)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if ctx_len.dtype != torch.int32 or not ctx_len.is_cuda:
        raise ValueError("ctx_len must be an int32 CUDA tensor")
    B, L, Hkv, D = k_blk.shape
    if tuple(v_blk.shape) != (B, L, Hkv, D) or k_ctx.shape[:2] != (B, Hkv) or \
            k_ctx.shape[3] != D or tuple(v_ctx.shape) != tuple(k_ctx.shape):
        raise ValueError("kv_append: inconsistent shapes")
    h = h or handle(k_blk.device.index)
    desc = AttnDesc(B, L, Hkv, Hkv, D, int(k_ctx.shape[2]), 0.0)
    _check(lib().tt_kv_append(h.ptr, ctypes.byref(desc), _dev_ptr(k_blk), _dev_ptr(v_blk),
                              _dev_ptr(k_ctx), _dev_ptr(v_ctx), _dev_ptr(ctx_len),
                              _stream_ptr(k_blk, stream)), "tt_kv_append")
    return k_ctx, v_ctx


def _check_commit_args(logits, masked, tok):
    import torch
    if logits.dtype != torch.float32 or not logits.is_cuda or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous CUDA float32 tensor")
    if masked.dtype != torch.uint8 or tok.dtype != torch.int32:
        raise ValueError("masked must be uint8 and tok int32")


def commit(logits, B: int, L: int, masked, k: int, tok, masked_out=None,
           h: Handle | None = None, stream=None):
    """One unmask/commit step (Algorithm 2, budget k per block).

    logits [B*L][V] float32, masked [B*L] uint8, tok [B*L] int32 (updated in
    place at committed rows). ``masked_out`` may be ``masked`` itself (in
    place). Returns (tok, masked_out).
    """
    import torch
    _check_commit_args(logits, masked, tok)
    h = h or handle(logits.device.index)
    if masked_out is None:
        masked_out = torch.empty_like(masked)
    _check(lib().tt_commit(h.ptr, _dev_ptr(logits), int(B), int(L), int(logits.shape[1]),
                           _dev_ptr(masked), int(k), _dev_ptr(tok), _dev_ptr(masked_out),
                           _stream_ptr(logits, stream)), "tt_commit")
    return tok, masked_out


def commit_threshold(logits, B: int, L: int, masked, gamma: float, steps_left: int, tok,
                     masked_out=None, h: Handle | None = None, stream=None):
    """One threshold unmasking step (Algorithm 2): per block, every masked row
    whose confidence is above gamma, and at least ceil(#masked / steps_left).

    Arguments and results as :func:`commit`.
    """
    import torch
    _check_commit_args(logits, masked, tok)
    h = h or handle(logits.device.index)
    if masked_out is None:
        masked_out = torch.empty_like(masked)
    _check(lib().tt_commit_threshold(h.ptr, _dev_ptr(logits), int(B), int(L), int(logits.shape[1]),
                                     _dev_ptr(masked), float(gamma), int(steps_left), _dev_ptr(tok),
                                     _dev_ptr(masked_out), _stream_ptr(logits, stream)),
           "tt_commit_threshold")
    return tok, masked_out


def commit_keys(rows: int, h: Handle | None = None, device=None, stream=None):
    """(key[rows] as int64 bits, arg[rows] int32) of the last commit call on the
    handle (tt_commit_keys), as new device tensors."""
    import torch
    h = h or handle(device)
    dev = torch.device("cuda", h.device)
    keys = torch.empty(rows, dtype=torch.int64, device=dev)
    args = torch.empty(rows, dtype=torch.int32, device=dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(lib().tt_commit_keys(h.ptr, _dev_ptr(keys), _dev_ptr(args), int(rows),
                                ctypes.c_void_p(st.cuda_stream)), "tt_commit_keys")
    return keys, args


def lm_head(hidden, weight, logits=None, h: Handle | None = None, stream=None):
    """The denoiser's LM head: logits = hidden @ weight^T (bf16 in, fp32 out) on
    the tensor core; each row's maximum and prediction stay in the handle for
    :func:`commit_rowmax`. hidden [M][K], weight [V][K] (torch.bfloat16, CUDA,
    contiguous). Returns logits [M][V] float32."""
    import torch
    for name, t in (("hidden", hidden), ("weight", weight)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    M, K = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != K:
        raise ValueError("lm_head: hidden and weight disagree on K")
    h = h or handle(hidden.device.index)
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=hidden.device)
    _check(lib().tt_lm_head(h.ptr, _dev_ptr(hidden), _dev_ptr(weight), int(M), int(K), int(V),
                            _dev_ptr(logits), _stream_ptr(hidden, stream)), "tt_lm_head")
    return logits


def commit_rowmax(logits, B: int, L: int, masked, k: int, tok, masked_out=None,
                  h: Handle | None = None, stream=None):
    """The commit step on the logits of the last :func:`lm_head` call on the
    handle, with the row maxima it found (tt_commit_rowmax). Arguments and
    results as :func:`commit`."""
    import torch
    _check_commit_args(logits, masked, tok)
    h = h or handle(logits.device.index)
    if masked_out is None:
        masked_out = torch.empty_like(masked)
    _check(lib().tt_commit_rowmax(h.ptr, _dev_ptr(logits), int(B), int(L), int(logits.shape[1]),
                                  _dev_ptr(masked), int(k), _dev_ptr(tok), _dev_ptr(masked_out),
                                  _stream_ptr(logits, stream)), "tt_commit_rowmax")
    return tok, masked_out
