"""GPU parity of tt_block_attn against the fp64 CPU oracle.

Block attention, "Nemotron-Labs-TwoTower" Section 2.1, Eq. (1). Acceptance:
max |gpu - oracle| <= 1e-2 * max |oracle| over the compared outputs (bf16
inputs, fp32 accumulation, bf16 output). Positions of the context cache at or
past ctx_len hold NaN, so any read of them fails the test.
"""
import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module")
def tt():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_decoding_attn_b300 as tt
    from block_diffusion_decoding_attn_b300 import build
    build.build()
    return tt


def _run_gpu(tt, inp, **kw):
    import torch
    t = wl.attn_tensors(inp)
    out = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"], **kw)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    return out.float().cpu().numpy().astype(np.float64), t


def _assert_close(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    bound = TOL * np.abs(ref).max()
    assert err <= bound, (err, bound)


SMALL = [
    # name, B, L, Hq, Hkv, D, cap, ctx, qk_std
    ("ragged_gqa4_d128", 2, 40, 8, 2, 128, 700, (300, 517), 0.0),
    ("gqa16_d128_two_mtiles", 2, 17, 32, 2, 128, 260, (129, 256), 0.0),
    ("d64_gqa4", 3, 32, 4, 1, 64, 300, (256, 1, 300), 0.0),
    ("empty_ctx", 2, 24, 8, 1, 128, 128, (0, 0), 0.0),
    ("block_of_one", 3, 1, 16, 1, 128, 1000, (999, 640, 1), 0.0),
    ("long_block_two_tiles", 1, 200, 4, 2, 128, 384, (384,), 0.0),
    ("mha_g1", 1, 64, 2, 2, 64, 130, (130,), 0.0),
    ("sharp_scores", 2, 32, 16, 1, 128, 1024, (1000, 333), 1.0),
    ("sharp_d64", 1, 48, 8, 2, 64, 777, (777,), 1.0),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases(tt, oracle_lib, case):
    name, B, L, Hq, Hkv, D, cap, ctx, qk = case
    w = wl.custom(name, B, L, Hq, Hkv, D, cap, ctx, qk_std=qk)
    inp = wl.attn_inputs(w, seed=1)
    got, _ = _run_gpu(tt, inp)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_splits_merge(tt, oracle_lib, splits):
    w = wl.custom("splits", 2, 32, 16, 2, 128, 1100, (1100, 45), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=2)
    got, _ = _run_gpu(tt, inp, num_splits=splits)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


def test_cache_is_not_modified(tt):
    import torch
    w = wl.custom("const_cache", 2, 16, 8, 2, 128, 300, (300, 200))
    inp = wl.attn_inputs(w, seed=3, pad=wl.to_bf16_bits(np.float32([7.0]))[0])
    t = wl.attn_tensors(inp)
    before = (t["k_ctx"].view(torch.int16).sum().item(), t["v_ctx"].view(torch.int16).sum().item())
    tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"],
                  num_splits=2)
    torch.cuda.synchronize()
    after = (t["k_ctx"].view(torch.int16).sum().item(), t["v_ctx"].view(torch.int16).sum().item())
    assert before == after


def test_ctx_len_out_of_range_is_flagged(tt):
    import torch
    w = wl.custom("bad_len", 1, 8, 4, 1, 64, 128, (128,))
    inp = wl.attn_inputs(w, seed=4)
    t = wl.attn_tensors(inp)
    t["ctx_len"].fill_(500)
    tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"])
    torch.cuda.synchronize()
    assert tt.handle().get_error() & tt.TT_DEV_CTX_LEN_RANGE
    assert tt.handle().get_error() == 0  # cleared by the read


def _sample_rows(w, ctx, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, w.B, n), rng.integers(0, w.L, n), rng.integers(0, w.Hq, n)], 1)
    # always include the longest and the shortest sequence, first and last position
    bl, bs = int(np.argmax(ctx)), int(np.argmin(ctx))
    extra = np.array([[bl, 0, 0], [bl, w.L - 1, w.Hq - 1], [bs, 0, w.Hq - 1], [bs, w.L - 1, 0]])
    return np.concatenate([rows, extra]).astype(np.int32)


@pytest.mark.parametrize("name", ["tiny_c256_l32", "b8_c4096_l32", "b16_c1024_l256"])
def test_full_workloads_all_rows(tt, oracle_lib, name):
    w = wl.WORKLOADS[name]
    inp = wl.attn_inputs(w, seed=0)
    got, _ = _run_gpu(tt, inp)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


def test_gen8k_schedule_sampled(tt, oracle_lib):
    w = wl.WORKLOADS["b4_gen8k_32x256"]
    for call in (0, 13, 31):
        inp = wl.attn_inputs(w, seed=0, call=call)
        got, _ = _run_gpu(tt, inp)
        assert np.isfinite(got).all()
        rows = _sample_rows(w, inp.ctx_len, 48, call)
        ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx,
                                    inp.ctx_len, rows=rows)
        _assert_close(got[rows[:, 0], rows[:, 1], rows[:, 2]], ref)


def test_ragged_long_context_sampled(tt, oracle_lib):
    w = wl.WORKLOADS["b64_ragged8k32k_l64"]
    inp = wl.attn_inputs(w, seed=0)
    got, _ = _run_gpu(tt, inp)
    assert np.isfinite(got).all()
    rows = _sample_rows(w, inp.ctx_len, 96, 7)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len,
                                rows=rows)
    _assert_close(got[rows[:, 0], rows[:, 1], rows[:, 2]], ref)
