"""GPU parity of the context-tower update: tt_block_attn_causal and tt_kv_append.

"Nemotron-Labs-TwoTower" Section 2.1, Algorithm 1 (the context update after a commit): the
committed block's tokens run causally over the prefix cache (query l sees the
cache and block keys 0..l), then the block's keys/values join the cache.
Acceptance: attention within 1e-2 * max |oracle| (as for tt_block_attn); the
append bit-exact, with blocks that do not fit left untouched and flagged.
Cache positions at or past ctx_len hold NaN, so any read of them fails.
"""
import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl
from conftest import KERNELS, attn_schedule

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
    out = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"],
                        causal=True, **kw)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    return out.float().cpu().numpy().astype(np.float64)


def _oracle(o, inp, **kw):
    return o.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len,
                        causal=True, **kw)


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
    ("empty_ctx_two_block_tiles", 1, 256, 2, 1, 128, 128, (0,), 0.0),
    ("block_of_one", 3, 1, 16, 1, 128, 1000, (999, 640, 1), 0.0),
    ("long_block_two_tiles", 1, 200, 4, 2, 128, 384, (384,), 0.0),
    ("mha_g1_d64", 1, 130, 2, 2, 64, 130, (77,), 0.0),
    ("sharp_scores", 2, 32, 16, 1, 128, 1024, (1000, 333), 1.0),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases(tt, oracle_lib, case):
    name, B, L, Hq, Hkv, D, cap, ctx, qk = case
    w = wl.custom(name, B, L, Hq, Hkv, D, cap, ctx, qk_std=qk)
    inp = wl.attn_inputs(w, seed=1)
    _assert_close(_run_gpu(tt, inp), _oracle(oracle_lib, inp))


@pytest.mark.parametrize("sched", [(0, 0, 0, 0), (2, 1, 1, 0), (2, 2, 1, 0), (2, 3, 1, 0), (2, 0, 1, 0),
                                   (1, 0, 0, 2), (1, 0, 0, 3), (1, 0, 0, 5)])
def test_cut_pieces_with_fully_masked_tiles(tt, oracle_lib, sched):
    # 3 context tiles + 2 block tiles per unit: with one-tile pieces, a piece
    # holding only block keys 128..199 has no key that rows l < 128 may see
    # (m = -inf there); the merge gives it weight 0.
    w = wl.custom("splits", 2, 200, 4, 2, 128, 384, (384, 300), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=2)
    with attn_schedule(tt, *sched):
        got = _run_gpu(tt, inp)
    _assert_close(got, _oracle(oracle_lib, inp))


def test_no_context_one_piece_per_block_tile(tt, oracle_lib):
    w = wl.custom("blk_only", 2, 256, 8, 1, 64, 128, (0, 0), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=3)
    ref = _oracle(oracle_lib, inp)
    for sched in ((2, 0, 1, 0), (1, 0, 0, 2)):
        with attn_schedule(tt, *sched):
            got = _run_gpu(tt, inp)
        _assert_close(got, ref)


def test_last_row_matches_bidirectional_call(tt):
    import torch
    w = wl.custom("last", 2, 48, 16, 1, 128, 600, (600, 222), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=4)
    t = wl.attn_tensors(inp)
    ca = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"],
                       causal=True)
    bi = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"])
    torch.cuda.synchronize()
    assert torch.equal(ca[:, -1], bi[:, -1])
    assert not torch.equal(ca[:, 0], bi[:, 0])


def test_full_workload_l256_all_rows(tt, oracle_lib):
    w = wl.WORKLOADS["b16_c1024_l256"]
    inp = wl.attn_inputs(w, seed=0)
    _assert_close(_run_gpu(tt, inp), _oracle(oracle_lib, inp))


def test_gen8k_schedule_every_call_all_rows(tt, oracle_lib):
    # the context tower's pass over each of the 32 committed blocks
    w = wl.WORKLOADS["b4_gen8k_32x256"]
    for call in range(len(w.ctx_schedule)):
        inp = wl.attn_inputs(w, seed=0, call=call)
        ref = _oracle(oracle_lib, inp)
        for sched in KERNELS:
            with attn_schedule(tt, *sched):
                got = _run_gpu(tt, inp)
            _assert_close(got, ref)


# ---------------------------------------------------------------- K/V append

def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("D", [64, 128])
def test_append_bit_exact_with_overflow(tt, oracle_lib, D):
    import torch
    B, L, Hkv, cap = 5, 40, 2, 300
    rng = np.random.default_rng(D)
    k_blk = rng.integers(0, 2**16, (B, L, Hkv, D), dtype=np.uint16)
    v_blk = rng.integers(0, 2**16, (B, L, Hkv, D), dtype=np.uint16)
    k_ctx = rng.integers(0, 2**16, (B, Hkv, cap, D), dtype=np.uint16)
    v_ctx = rng.integers(0, 2**16, (B, Hkv, cap, D), dtype=np.uint16)
    ctx_len = np.array([0, 137, 260, 261, 300], np.int32)  # 260 fits exactly; 261, 300 do not
    ek, ev, en, fits = oracle_lib.kv_append(k_blk, v_blk, k_ctx, v_ctx, ctx_len)
    assert list(fits) == [True, True, True, False, False]

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    tk, tv, tkc, tvc = dev(k_blk), dev(v_blk), dev(k_ctx), dev(v_ctx)
    tn = torch.from_numpy(ctx_len).cuda()
    tt.kv_append(tk, tv, tkc, tvc, tn)
    torch.cuda.synchronize()
    assert tt.handle().get_error() & tt.TT_DEV_CTX_LEN_RANGE
    np.testing.assert_array_equal(_bits(tkc), ek)
    np.testing.assert_array_equal(_bits(tvc), ev)
    np.testing.assert_array_equal(tn.cpu().numpy(), en)
    np.testing.assert_array_equal(_bits(tk), k_blk)  # the block is only read


def test_append_then_decode_rows_match_causal_pass(tt, oracle_lib):
    # The update as a whole: the causal pass over (cache, block), then the block
    # joins the cache; a bidirectional one-token call for the last block token
    # over the cache holding tokens 0..L-2 equals the causal pass's last row.
    import torch
    w = wl.custom("update", 2, 32, 16, 2, 128, 512, (300, 111), qk_std=0.5)
    inp = wl.attn_inputs(w, seed=6)
    t = wl.attn_tensors(inp)
    causal = tt.block_attn(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], t["ctx_len"],
                           causal=True)
    n = t["ctx_len"].clone()
    tt.kv_append(t["k_blk"][:, :-1].contiguous(), t["v_blk"][:, :-1].contiguous(), t["k_ctx"],
                 t["v_ctx"], n)
    one = tt.block_attn(t["q"][:, -1:].contiguous(), t["k_blk"][:, -1:].contiguous(),
                        t["v_blk"][:, -1:].contiguous(), t["k_ctx"], t["v_ctx"], n)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    assert torch.equal(n.cpu(), torch.tensor([300 + 31, 111 + 31], dtype=torch.int32))
    ref = _oracle(oracle_lib, inp)
    _assert_close(one[:, 0].float().cpu().numpy().astype(np.float64), ref[:, -1])
    _assert_close(causal[:, -1].float().cpu().numpy().astype(np.float64), ref[:, -1])


def test_append_invalid_arguments_raise(tt):
    import torch
    k = torch.zeros(1, 4, 1, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 1, 3, 64, dtype=torch.bfloat16, device="cuda")  # cap 3 < L 4
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tt.TTError):
        tt.kv_append(k, k, kc, kc, n)
