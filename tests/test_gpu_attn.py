"""GPU parity of tt_block_attn against the fp64 CPU oracle.

Block attention, "Nemotron-Labs-TwoTower" Section 2.1, Eq. (1). Acceptance:
max |gpu - oracle| <= 1e-2 * max |oracle| over the compared outputs (bf16
inputs, fp32 accumulation, bf16 output). Positions of the context cache at or
past ctx_len hold NaN, so any read of them fails the test.
"""
import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl
from conftest import KERNELS, SCHEDULES, attn_schedule

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


EXTREME = [
    # the largest query group, Hq/Hkv = 128: one block position per 128-row
    # query tile, and an odd tile count (a pair with one tile)
    ("gqa128_max_group", 2, 3, 128, 1, 64, 200, (200, 57), 0.0),
    # a long block: 9 block KV tiles, the last one partial, and 18 query tiles
    ("long_block_nine_tiles", 1, 1100, 4, 2, 128, 300, (300,), 0.0),
]


@pytest.mark.parametrize("sched", KERNELS, ids=["per_unit", "persistent"])
@pytest.mark.parametrize("causal", [False, True], ids=["bidirectional", "causal"])
@pytest.mark.parametrize("case", EXTREME, ids=[c[0] for c in EXTREME])
def test_extreme_shapes(tt, oracle_lib, case, causal, sched):
    name, B, L, Hq, Hkv, D, cap, ctx, qk = case
    w = wl.custom(name, B, L, Hq, Hkv, D, cap, ctx, qk_std=qk)
    inp = wl.attn_inputs(w, seed=3)
    with attn_schedule(tt, *sched):
        got, _ = _run_gpu(tt, inp, causal=causal)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len,
                                causal=causal)
    _assert_close(got, ref)


@pytest.mark.parametrize("sched", KERNELS, ids=["per_unit", "persistent"])
def test_two_million_position_context(tt, oracle_lib, sched):
    # a 2^21-position cache, all but 3 positions filled, behind an 8-token
    # block: the one-unit-per-CTA schedule splits the one unit 64 ways, the
    # persistent one cuts its query tile into one piece per SM and merges them
    # in the kernel
    w = wl.custom("ctx2m", 1, 8, 4, 1, 64, 1 << 21, ((1 << 21) - 3,))
    inp = wl.attn_inputs(w, seed=4)
    with attn_schedule(tt, *sched):
        got, _ = _run_gpu(tt, inp)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


@pytest.mark.parametrize("sched", SCHEDULES)
def test_schedules_cut_and_merge(tt, oracle_lib, sched):
    # query tiles cut between CTAs at every tile boundary, merged by the last piece
    w = wl.custom("splits", 2, 32, 16, 2, 128, 1100, (1100, 45), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=2)
    with attn_schedule(tt, *sched):
        got, _ = _run_gpu(tt, inp)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


@pytest.mark.parametrize("sched", [(2, 0, 1, 0), (2, 5, 1, 0), (2, 12, 2, 0), (1, 0, 0, 0), (1, 0, 0, 3)])
def test_schedules_pair_groups(tt, oracle_lib, sched):
    # 8 query tiles per (b, kv head): pair blocks of several CTAs, ragged lengths
    w = wl.custom("groups", 3, 64, 32, 2, 128, 900, (900, 3, 517), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=6)
    with attn_schedule(tt, *sched):
        got, _ = _run_gpu(tt, inp)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    _assert_close(got, ref)


def test_deterministic_under_one_schedule(tt):
    w = wl.custom("det", 2, 32, 16, 2, 128, 1100, (1100, 45), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=2)
    for sched in ((2, 0, 1, 0), (1, 0, 0, 3)):
        with attn_schedule(tt, *sched):
            a, _ = _run_gpu(tt, inp)
            b, _ = _run_gpu(tt, inp)
        assert np.array_equal(a, b)


def test_cache_is_not_modified(tt):
    import torch
    w = wl.custom("const_cache", 2, 16, 8, 2, 128, 300, (300, 200))
    inp = wl.attn_inputs(w, seed=3, pad=wl.to_bf16_bits(np.float32([7.0]))[0])
    t = wl.attn_tensors(inp)
    before = (t["k_ctx"].view(torch.int16).sum().item(), t["v_ctx"].view(torch.int16).sum().item())
    for sched in ((2, 0, 1, 0), (1, 0, 0, 2)):
        with attn_schedule(tt, *sched):
            tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"])
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


@pytest.mark.parametrize("name", ["tiny_c256_l32", "b8_c4096_l32", "b16_c1024_l256",
                                  "b64_ragged8k32k_l64"])
def test_full_workloads_all_rows(tt, oracle_lib, name):
    # every output row against the oracle, with each of the two schedules
    w = wl.WORKLOADS[name]
    inp = wl.attn_inputs(w, seed=0)
    ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    for sched in KERNELS:
        with attn_schedule(tt, *sched):
            got, _ = _run_gpu(tt, inp)
        _assert_close(got, ref)


def test_gen8k_schedule_every_call_all_rows(tt, oracle_lib):
    # the 32 calls of the 8K-token generation (context 1024, 1280, ..., 8960)
    w = wl.WORKLOADS["b4_gen8k_32x256"]
    for call in range(len(w.ctx_schedule)):
        inp = wl.attn_inputs(w, seed=0, call=call)
        ref = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx,
                                    inp.ctx_len)
        for sched in KERNELS:
            with attn_schedule(tt, *sched):
                got, _ = _run_gpu(tt, inp)
            _assert_close(got, ref)
