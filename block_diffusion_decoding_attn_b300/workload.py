"""Seeded synthetic inputs for one TwoTower denoising step.

This module only draws and lays out numbers. It holds none of the method's
arithmetic (no attention, no softmax, no commit rule), so both the CPU oracle
and the CUDA path can take their inputs from it.

Shapes follow the denoising-step hot path of "Nemotron-Labs-TwoTower:
Diffusion Language Modeling with Pretrained Autoregressive Context"
(Section 2.1, Eq. 1 block attention; Section 2.2, Algorithm 2 confidence
unmasking):

* q      [B][L][Hq][D]         bf16   queries of the noisy block
* k_blk  [B][L][Hkv][D]        bf16   denoiser's own keys for the block
* v_blk  [B][L][Hkv][D]        bf16
* k_ctx  [B][Hkv][C_cap][D]    bf16   context-tower KV cache of the same layer
* v_ctx  [B][Hkv][C_cap][D]    bf16
* ctx_len[B]                   int32  valid context positions per sequence
* logits [B*L][V]              fp32   denoiser vocabulary logits
* masked [B*L]                 uint8  1 = position still [MASK]
* tok    [B*L]                 int32  committed ids (-1 = [MASK])

Values: Q/K/V are N(0,1)/sqrt(D) drawn in fp32 and rounded to bf16
(round-to-nearest-even); logits are N(0, 4) (variance 4, sigma 2). Context
positions at or beyond ctx_len[b] hold a sentinel (a NaN pattern by default)
so that any read of them shows up in the output.

Random numbers come from numpy's Philox4x32-10 bit generator, keyed by
(seed, workload id, tensor id, chunk index), so the result does not depend on
the thread count used to fill it.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Tensor ids in the Philox key.
_T_Q, _T_KBLK, _T_VBLK, _T_KCTX, _T_VCTX, _T_LOGITS, _T_CTXLEN = 1, 2, 3, 4, 5, 6, 7
_T_HIDDEN, _T_WEIGHT = 8, 9

# Input width of the denoiser's LM head. The pages name the backbone
# (Nemotron-3-Nano-30B-A3B) but not its hidden size; 2688 is read as that
# backbone's hidden size.
LM_HIDDEN = 2688

_CHUNK = 1 << 22  # elements per independently keyed chunk

BF16_NAN = np.uint16(0x7FC0)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One denoising-step workload: shapes, value recipe and commit budget."""
    name: str
    wid: int            # workload id in the Philox key
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    ctx_cap: int
    V: int
    k: int              # positions committed per block per step
    ctx: tuple = ()     # fixed ctx_len per sequence; empty => drawn
    ctx_range: tuple = ()  # (lo, hi) inclusive uniform integer draw
    ctx_schedule: tuple = ()  # per-call ctx_len (one attention call per block)
    qk_std: float = 0.0  # 0 => 1/sqrt(D)
    logit_std: float = 2.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def rows(self) -> int:
        return self.B * self.L

    @property
    def steps_to_unmask(self) -> int:
        return -(-self.L // self.k)


# The five workloads. Names say what each is; sizes as stated.
WORKLOADS = {
    "tiny_c256_l32": Workload(
        "tiny_c256_l32", 0, B=1, L=32, Hq=4, Hkv=1, D=64, ctx_cap=256, V=1024, k=4,
        ctx=(256,)),
    "b8_c4096_l32": Workload(
        "b8_c4096_l32", 1, B=8, L=32, Hq=32, Hkv=2, D=128, ctx_cap=4096, V=131072, k=4,
        ctx=(4096,) * 8),
    "b16_c1024_l256": Workload(
        "b16_c1024_l256", 2, B=16, L=256, Hq=32, Hkv=2, D=128, ctx_cap=1024, V=131072, k=16,
        ctx=(1024,) * 16),
    "b4_gen8k_32x256": Workload(
        "b4_gen8k_32x256", 3, B=4, L=256, Hq=32, Hkv=2, D=128, ctx_cap=8960, V=131072, k=32,
        ctx_schedule=tuple(1024 + 256 * j for j in range(32))),
    "b64_ragged8k32k_l64": Workload(
        "b64_ragged8k32k_l64", 4, B=64, L=64, Hq=32, Hkv=2, D=128, ctx_cap=32768, V=131072, k=8,
        ctx_range=(8192, 32768)),
}

WORKLOAD_ORDER = list(WORKLOADS)


def custom(name: str, B: int, L: int, Hq: int, Hkv: int, D: int, ctx_cap: int,
           ctx, V: int = 1024, k: int = 4, wid: int = 100, qk_std: float = 0.0,
           logit_std: float = 2.0) -> Workload:
    """A test-sized workload with explicit per-sequence ctx_len."""
    return Workload(name, wid, B=B, L=L, Hq=Hq, Hkv=Hkv, D=D, ctx_cap=ctx_cap, V=V,
                    k=k, ctx=tuple(int(c) for c in ctx), qk_std=qk_std,
                    logit_std=logit_std)


def _rng(seed: int, wid: int, tid: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, wid, tid, chunk])))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill_normal(n: int, std: float, seed: int, wid: int, tid: int, bf16: bool) -> np.ndarray:
    """n draws of N(0, std^2), chunk-keyed; bf16 bit patterns or fp32."""
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    nchunks = max(1, -(-n // _CHUNK))

    def work(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        tmp = np.empty(hi - lo, dtype=np.float32)
        _rng(seed, wid, tid, c).standard_normal(out=tmp, dtype=np.float32)
        tmp *= np.float32(std)
        out[lo:hi] = to_bf16_bits(tmp) if bf16 else tmp

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def ctx_lens(w: Workload, seed: int = 0, call: int = 0) -> np.ndarray:
    """ctx_len[B] for attention call `call` (only schedules have >1 call)."""
    if w.ctx_schedule:
        return np.full(w.B, w.ctx_schedule[call], dtype=np.int32)
    if w.ctx_range:
        lo, hi = w.ctx_range
        return _rng(seed, w.wid, _T_CTXLEN, 0).integers(lo, hi + 1, size=w.B).astype(np.int32)
    return np.asarray(w.ctx, dtype=np.int32)


def num_calls(w: Workload) -> int:
    return len(w.ctx_schedule) if w.ctx_schedule else 1


@dataclasses.dataclass
class AttnInputs:
    q: np.ndarray       # uint16 bf16 bits [B][L][Hq][D]
    k_blk: np.ndarray   # uint16 [B][L][Hkv][D]
    v_blk: np.ndarray
    k_ctx: np.ndarray   # uint16 [B][Hkv][C_cap][D]
    v_ctx: np.ndarray
    ctx_len: np.ndarray  # int32 [B]
    scale: float


def attn_inputs(w: Workload, seed: int = 0, call: int = 0, pad=BF16_NAN) -> AttnInputs:
    """Inputs of attention call `call`; `pad` fills ctx positions >= ctx_len."""
    std = w.qk_std if w.qk_std > 0 else 1.0 / math.sqrt(w.D)
    B, L, Hq, Hkv, D, C = w.B, w.L, w.Hq, w.Hkv, w.D, w.ctx_cap
    # Blocks of a multi-call schedule get fresh Q / block K / block V.
    sub = call * 16
    q = _fill_normal(B * L * Hq * D, std, seed, w.wid, _T_Q + sub, True).reshape(B, L, Hq, D)
    kb = _fill_normal(B * L * Hkv * D, std, seed, w.wid, _T_KBLK + sub, True).reshape(B, L, Hkv, D)
    vb = _fill_normal(B * L * Hkv * D, std, seed, w.wid, _T_VBLK + sub, True).reshape(B, L, Hkv, D)
    # The context cache is filled once for the whole schedule.
    kc = _fill_normal(B * Hkv * C * D, std, seed, w.wid, _T_KCTX, True).reshape(B, Hkv, C, D)
    vc = _fill_normal(B * Hkv * C * D, std, seed, w.wid, _T_VCTX, True).reshape(B, Hkv, C, D)
    cl = ctx_lens(w, seed, call)
    if pad is not None:
        for b in range(B):
            kc[b, :, cl[b]:, :] = pad
            vc[b, :, cl[b]:, :] = pad
    return AttnInputs(q, kb, vb, kc, vc, cl, 1.0 / math.sqrt(D))


def block_inputs(w: Workload, seed: int = 0, call: int = 0):
    """q, k_blk, v_blk of attention call `call` alone (the draws attn_inputs
    makes for them), for schedules that share one context cache."""
    std = w.qk_std if w.qk_std > 0 else 1.0 / math.sqrt(w.D)
    B, L, Hq, Hkv, D = w.B, w.L, w.Hq, w.Hkv, w.D
    sub = call * 16
    q = _fill_normal(B * L * Hq * D, std, seed, w.wid, _T_Q + sub, True).reshape(B, L, Hq, D)
    kb = _fill_normal(B * L * Hkv * D, std, seed, w.wid, _T_KBLK + sub, True).reshape(B, L, Hkv, D)
    vb = _fill_normal(B * L * Hkv * D, std, seed, w.wid, _T_VBLK + sub, True).reshape(B, L, Hkv, D)
    return q, kb, vb


@dataclasses.dataclass
class CommitInputs:
    logits: np.ndarray  # float32 [B*L][V]
    masked: np.ndarray  # uint8 [B*L]
    tok: np.ndarray     # int32 [B*L]
    k: int


def logits(w: Workload, seed: int = 0, step: int = 0) -> np.ndarray:
    return _fill_normal(w.rows * w.V, w.logit_std, seed, w.wid, _T_LOGITS + 16 * step,
                        False).reshape(w.rows, w.V)


def commit_inputs(w: Workload, seed: int = 0, step: int = 0) -> CommitInputs:
    """Step-`step` logits over a fully masked block (step 0 = first step)."""
    return CommitInputs(logits(w, seed, step), np.ones(w.rows, dtype=np.uint8),
                        np.full(w.rows, -1, dtype=np.int32), w.k)


def random_mask(w: Workload, frac: float, seed: int = 0) -> np.ndarray:
    """A mask with about `frac` of the positions still masked (ragged per block)."""
    g = _rng(seed, w.wid, 99, 0)
    return (g.random(w.rows) < frac).astype(np.uint8)


def attn_tensors(inp: AttnInputs, device="cuda", pin: bool = False) -> dict:
    """The attention inputs as torch tensors (bf16 views of the bit patterns)."""
    import torch

    def t(a, bf16=True):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if bf16:
            x = x.view(torch.bfloat16)
        if pin:
            x = x.pin_memory()
        return x.to(device, non_blocking=pin) if device != "cpu" else x

    return dict(q=t(inp.q), k_blk=t(inp.k_blk), v_blk=t(inp.v_blk), k_ctx=t(inp.k_ctx),
                v_ctx=t(inp.v_ctx), ctx_len=t(inp.ctx_len, bf16=False))


def commit_tensors(inp: CommitInputs, device="cuda", pin: bool = False) -> dict:
    import torch

    def t(a):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if pin:
            x = x.pin_memory()
        return x.to(device, non_blocking=pin) if device != "cpu" else x

    return dict(logits=t(inp.logits), masked=t(inp.masked), tok=t(inp.tok))


def lm_head_inputs(M: int, K: int, V: int, seed: int = 0, wid: int = 200, step: int = 0):
    """hidden [M][K] ~ N(0, 1) and weight [V][K] ~ N(0, 4/K) as bf16 bit patterns,
    so that the logits hidden @ weight^T have variance about 4 (the logits'
    recipe, N(0, 4)). `step` draws a fresh hidden state (a later denoising step)."""
    hid = _fill_normal(M * K, 1.0, seed, wid, _T_HIDDEN + 16 * step, True).reshape(M, K)
    w = _fill_normal(V * K, 2.0 / math.sqrt(K), seed, wid, _T_WEIGHT, True).reshape(V, K)
    return hid, w


def _fill_int(n: int, lo: int, hi: int, scale: float, seed: int, wid: int, tid: int) -> np.ndarray:
    """n uniform integers in [lo, hi] times `scale` (a power of two), chunk-keyed,
    as bf16 bit patterns (exact: |integer| <= 256)."""
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, -(-n // _CHUNK))

    def work(c):
        a, b = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        v = _rng(seed, wid, tid, c).integers(lo, hi + 1, size=b - a).astype(np.float32)
        out[a:b] = to_bf16_bits(v * np.float32(scale))

    if nchunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def lm_head_exact_inputs(M: int, K: int, V: int, seed: int = 0, wid: int = 201, step: int = 0):
    """LM head inputs whose logits are exact in fp32 whatever the summation order:
    hidden [M][K] = i / 8 and weight [V][K] = j * 2^e with i, j uniform in
    [-8, 8] and 2^e the power of two nearest 2 / (3 sqrt K), so the logits have
    variance 9 K 2^(2e), between 1 and 16. Every product is a multiple of
    u = 2^(e-3) and every partial sum is at most 64 K u in magnitude, an integer
    count of u below 2^24 for K < 2^18: fp32 holds each one exactly, so an fp32
    accumulation in any order equals the exact sum (the logits of both the fp64
    LM head and the tensor-core one). Small integers also make ties among the
    logits and among the rows' confidences common."""
    if not 0 < K < 1 << 18:
        raise ValueError("lm_head_exact_inputs: K must be in [1, 2^18)")
    e = round(math.log2(2.0 / (3.0 * math.sqrt(K))))
    hid = _fill_int(M * K, -8, 8, 0.125, seed, wid, _T_HIDDEN + 16 * step).reshape(M, K)
    w = _fill_int(V * K, -8, 8, 2.0 ** e, seed, wid, _T_WEIGHT).reshape(V, K)
    return hid, w
