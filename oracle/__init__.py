"""Plain, slow CPU oracle for the TwoTower denoising-step hot path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only code allowed to import this package.
It shares no code with the CUDA path (no kernels, headers, helpers, tables or
constant generators); the two meet only in the seeded input generator
``block_diffusion_decoding_attn_b300.workload``, which holds none of the
method's arithmetic.

* ``block_attn`` follows "Nemotron-Labs-TwoTower" Section 2.1, Eq. (1): one
  softmax per query over [context keys; block keys], fp64, explicit loops
  (``attn_ref.c``).
* ``commit`` follows Section 2.2 / Algorithm 2 (confidence unmasking) with a
  fixed per-step budget k and the canonical fixed-point confidence key
  (``commit_ref.c``).
* ``block_attn_train`` follows Section 2.3, "Implementation": all noisy blocks
  of a clean sequence in one pass, block j attending to the clean positions
  before it and bidirectionally to itself (a loop over blocks of
  ``block_attn``).
* ``lm_head`` is the denoiser's output layer before Section 2.2's sampling:
  logits = hidden @ weight^T over bf16 values, in float64.
* ``block_attn(..., causal=True)`` and ``kv_append`` follow Section 2.1,
  Algorithm 1 (the context update after a commit): the context tower's causal pass over a
  committed block, and its keys/values joining the prefix cache.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, "attn_ref.c"), os.path.join(_HERE, "commit_ref.c")]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fp contraction: fmaf is called explicitly)."""
    newest = max(os.path.getmtime(s) for s in _SRC)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp] + _SRC + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.tt_oracle_block_attn.restype = ctypes.c_int
            lib.tt_oracle_block_attn.argtypes = [ctypes.c_int] * 6 + [ctypes.c_double] + [P] * 6 + [
                ctypes.c_int, P, P, ctypes.c_int]
            lib.tt_oracle_block_attn_causal.restype = ctypes.c_int
            lib.tt_oracle_block_attn_causal.argtypes = lib.tt_oracle_block_attn.argtypes
            lib.tt_oracle_exp_own.restype = ctypes.c_float
            lib.tt_oracle_exp_own.argtypes = [ctypes.c_float]
            lib.tt_oracle_exp_n.restype = ctypes.c_float
            lib.tt_oracle_exp_n.argtypes = [ctypes.c_float]
            lib.tt_oracle_quant.restype = ctypes.c_uint64
            lib.tt_oracle_quant.argtypes = [ctypes.c_float]
            lib.tt_oracle_row_key.restype = None
            lib.tt_oracle_row_key.argtypes = [P, ctypes.c_long, P, P]
            lib.tt_oracle_commit.restype = ctypes.c_int
            lib.tt_oracle_commit.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_long, P,
                                             ctypes.c_int, P, P, P, P, ctypes.c_int]
            lib.tt_oracle_conf_above.restype = ctypes.c_int
            lib.tt_oracle_conf_above.argtypes = [ctypes.c_uint64, ctypes.c_double]
            lib.tt_oracle_commit_threshold.restype = ctypes.c_int
            lib.tt_oracle_commit_threshold.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                                       P, ctypes.c_double, ctypes.c_int, P, P, P, P,
                                                       ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def block_attn(q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, scale=None, rows=None, threads=0,
               causal=False):
    """fp64 block attention (Eq. 1); ``causal``: block query l sees block keys 0..l only.

    q [B][L][Hq][D], k_blk/v_blk [B][L][Hkv][D], k_ctx/v_ctx [B][Hkv][C_cap][D]
    as bf16 bit patterns (uint16); ctx_len [B] int32. ``scale`` None means
    1/sqrt(D). ``rows`` None gives the full [B][L][Hq][D] output; otherwise an
    [n][3] int array of (b, l, h) triples and an [n][D] output.
    """
    lib = _load()
    q, k_blk, v_blk = _c(q, np.uint16), _c(k_blk, np.uint16), _c(v_blk, np.uint16)
    k_ctx, v_ctx = _c(k_ctx, np.uint16), _c(v_ctx, np.uint16)
    ctx_len = _c(ctx_len, np.int32)
    B, L, Hq, D = q.shape
    Hkv, C = k_ctx.shape[1], k_ctx.shape[2]
    assert k_blk.shape == (B, L, Hkv, D) and v_blk.shape == k_blk.shape
    assert k_ctx.shape == (B, Hkv, C, D) and v_ctx.shape == k_ctx.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is None:
        out = np.empty((B, L, Hq, D), np.float64)
        n, rp = 0, None
    else:
        rows = _c(rows, np.int32).reshape(-1, 3)
        out = np.empty((rows.shape[0], D), np.float64)
        n, rp = rows.shape[0], _ptr(rows)
    fn = lib.tt_oracle_block_attn_causal if causal else lib.tt_oracle_block_attn
    rc = fn(B, L, Hq, Hkv, D, C, float(scale), _ptr(q), _ptr(k_blk), _ptr(v_blk), _ptr(k_ctx),
            _ptr(v_ctx), _ptr(ctx_len), n, rp, _ptr(out), int(threads))
    if rc != 0:
        raise ValueError("oracle block_attn: invalid arguments")
    return out


def block_attn_train(q, k_noisy, v_noisy, k_clean, v_clean, S, scale=None, rows=None, threads=0):
    """Training-time batched block attention (Section 2.3, "Implementation").

    q [B][N][Hq][D], k_noisy/v_noisy [B][N][Hkv][D], k_clean/v_clean [B][Hkv][N][D]
    (bf16 bit patterns). Noisy block j (tokens j*S .. j*S+S-1) of every sequence
    attends to [clean positions 0..j*S-1 ; its own S noisy tokens]: Eq. (1)
    with the clean sequence as the context cache and ctx_len = j*S. ``rows``
    None gives [B][N][Hq][D]; otherwise (b, n, h) triples and an [n][D] output.
    """
    q = _c(q, np.uint16)
    B, N, Hq, D = q.shape
    if S < 1 or N % S:
        raise ValueError("oracle block_attn_train: N must be a multiple of S")
    if rows is None:
        out = np.empty((B, N, Hq, D), np.float64)
        for j in range(N // S):
            sl = slice(j * S, (j + 1) * S)
            out[:, sl] = block_attn(q[:, sl], k_noisy[:, sl], v_noisy[:, sl], k_clean, v_clean,
                                    np.full(B, j * S, np.int32), scale=scale, threads=threads)
        return out
    rows = _c(rows, np.int32).reshape(-1, 3)
    out = np.empty((rows.shape[0], D), np.float64)
    for j in np.unique(rows[:, 1] // S):
        sel = np.nonzero(rows[:, 1] // S == j)[0]
        sub = rows[sel].copy()
        sub[:, 1] -= j * S
        sl = slice(j * S, (j + 1) * S)
        out[sel] = block_attn(q[:, sl], k_noisy[:, sl], v_noisy[:, sl], k_clean, v_clean,
                              np.full(B, j * S, np.int32), scale=scale, rows=sub, threads=threads)
    return out


def kv_append(k_blk, v_blk, k_ctx, v_ctx, ctx_len):
    """The cache after a committed block joins it (Section 2.1, Algorithm 1).

    k_blk/v_blk [B][L][Hkv][D], k_ctx/v_ctx [B][Hkv][C_cap][D] (any element
    type), ctx_len [B]. Returns new (k_ctx, v_ctx, ctx_len, fits): for every b
    with 0 <= ctx_len[b] <= C_cap - L, cache rows ctx_len[b] + l take block row
    l and ctx_len[b] grows by L; any other b is left as it was (fits[b] False).
    The inputs are not modified.
    """
    k_blk, v_blk = np.asarray(k_blk), np.asarray(v_blk)
    k_new, v_new = np.array(k_ctx, copy=True), np.array(v_ctx, copy=True)
    n_new = np.array(ctx_len, dtype=np.int64, copy=True)
    B, L, Hkv, D = k_blk.shape
    cap = k_new.shape[2]
    fits = np.zeros(B, dtype=bool)
    for b in range(B):
        c = int(n_new[b])
        if c < 0 or c + L > cap:
            continue
        fits[b] = True
        for l in range(L):
            for h in range(Hkv):
                k_new[b, h, c + l, :] = k_blk[b, l, h, :]
                v_new[b, h, c + l, :] = v_blk[b, l, h, :]
        n_new[b] = c + L
    return k_new, v_new, n_new.astype(np.int32), fits


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) widened exactly to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def lm_head(hidden, weight, rows=None):
    """The denoiser's LM head, the step that produces the vocabulary logits
    Section 2.2's sampling reads (Algorithm 2's distribution p_theta):
    logits[m][v] = sum_k hidden[m][k] * weight[v][k], in float64 over the bf16
    values (hidden [M][K], weight [V][K] as bf16 bit patterns). ``rows``: only
    those rows of hidden."""
    h = bf16_to_f64(hidden)
    if rows is not None:
        h = h[np.asarray(rows)]
    return h @ bf16_to_f64(weight).T


def exp_own(x: float) -> float:
    """The fp32 exponential that defines the canonical confidence key."""
    return _load().tt_oracle_exp_own(float(np.float32(x)))


def exp_n(x: float) -> int:
    """The integer n of the exponential's range reduction for x (x ~ n ln 2 + r)."""
    return int(_load().tt_oracle_exp_n(float(np.float32(x))))


def quant(x: float) -> int:
    """q(x) = rint(2^40 * e(x)) as an integer (0 below -30)."""
    return int(_load().tt_oracle_quant(float(np.float32(x))))


def row_key(row) -> tuple[int, int]:
    """(greedy prediction, canonical key) of one fp32 logit row."""
    lib = _load()
    row = _c(row, np.float32)
    a = np.zeros(1, np.int32)
    k = np.zeros(1, np.uint64)
    lib.tt_oracle_row_key(_ptr(row), row.shape[0], _ptr(a), _ptr(k))
    return int(a[0]), int(k[0])


def commit(logits, B, L, masked, k, tok, threads=0):
    """One confidence-unmasking step with budget k per block.

    Returns (tok_out, masked_out, keys, args); keys/args hold the key and
    prediction of each row that was masked on entry (0 elsewhere).
    """
    lib = _load()
    logits = _c(logits, np.float32)
    R, V = logits.shape
    assert R == B * L
    m_in = _c(masked, np.uint8).copy()
    tok_out = _c(tok, np.int32).copy()
    m_out = np.empty(R, np.uint8)
    keys = np.zeros(R, np.uint64)
    args = np.zeros(R, np.int32)
    rc = lib.tt_oracle_commit(_ptr(logits), B, L, V, _ptr(m_in), int(k), _ptr(tok_out),
                              _ptr(m_out), _ptr(keys), _ptr(args), int(threads))
    if rc != 0:
        raise ValueError("oracle commit: invalid arguments")
    return tok_out, m_out, keys, args


def conf_above(key: int, gamma: float) -> bool:
    """Whether a row with canonical key `key` has confidence 2^40/key > gamma (exact)."""
    return bool(_load().tt_oracle_conf_above(int(key), float(gamma)))


def commit_threshold(logits, B, L, masked, gamma, steps_left, tok, threads=0):
    """One threshold unmasking step (Algorithm 2): per block, every masked row
    with confidence > gamma, and at least ceil(#masked / steps_left) rows.

    Returns (tok_out, masked_out, keys, args) like ``commit``.
    """
    lib = _load()
    logits = _c(logits, np.float32)
    R, V = logits.shape
    assert R == B * L
    m_in = _c(masked, np.uint8).copy()
    tok_out = _c(tok, np.int32).copy()
    m_out = np.empty(R, np.uint8)
    keys = np.zeros(R, np.uint64)
    args = np.zeros(R, np.int32)
    rc = lib.tt_oracle_commit_threshold(_ptr(logits), B, L, V, _ptr(m_in), float(gamma),
                                        int(steps_left), _ptr(tok_out), _ptr(m_out), _ptr(keys),
                                        _ptr(args), int(threads))
    if rc != 0:
        raise ValueError("oracle commit_threshold: invalid arguments")
    return tok_out, m_out, keys, args
