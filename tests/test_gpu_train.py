"""GPU parity of tt_block_attn_train (training-time batched block attention).

"Nemotron-Labs-TwoTower" Section 2.3, "Implementation": every noisy block j of
a clean sequence attends to the clean positions 0..j*S-1 and bidirectionally to
its own S noisy tokens, all blocks in one call. Acceptance as for
tt_block_attn: max |gpu - oracle| <= 1e-2 * max |oracle|.
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


def _inputs(B, N, Hq, Hkv, D, seed, qk_std=0.0):
    w = wl.custom("train", B, N, Hq, Hkv, D, N, (N,) * B, qk_std=qk_std)
    return wl.attn_inputs(w, seed=seed)


def _run_gpu(tt, inp, S, **kw):
    import torch
    t = wl.attn_tensors(inp)
    out = tt.block_attn_train(t["q"], t["k_blk"], t["v_blk"], t["k_ctx"], t["v_ctx"], S, **kw)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    return out.float().cpu().numpy().astype(np.float64)


def _oracle(o, inp, S, **kw):
    return o.block_attn_train(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, S, **kw)


def _assert_close(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    bound = TOL * np.abs(ref).max()
    assert err <= bound, (err, bound)


SMALL = [
    # name, B, N, S, Hq, Hkv, D, qk_std
    ("s16_gqa16_d128", 2, 256, 16, 32, 2, 128, 0.0),
    ("s32_gqa4_d64", 1, 320, 32, 8, 2, 64, 0.0),
    ("s160_two_block_tiles", 2, 320, 160, 4, 1, 128, 0.0),
    ("s1_every_token_a_block", 2, 40, 1, 16, 1, 128, 0.0),
    ("one_block", 3, 64, 64, 8, 2, 128, 0.0),
    ("sharp_scores", 1, 512, 16, 16, 1, 128, 1.0),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases(tt, oracle_lib, case):
    name, B, N, S, Hq, Hkv, D, qk = case
    inp = _inputs(B, N, Hq, Hkv, D, seed=1, qk_std=qk)
    _assert_close(_run_gpu(tt, inp, S), _oracle(oracle_lib, inp, S))


@pytest.mark.parametrize("sched", [(2, 2, 1, 0), (2, 5, 1, 0), (2, 0, 1, 0), (1, 0, 0, 2), (1, 0, 0, 5)])
def test_cut_pieces(tt, oracle_lib, sched):
    inp = _inputs(2, 1024, 16, 2, 128, seed=2, qk_std=0.5)
    with attn_schedule(tt, *sched):
        got = _run_gpu(tt, inp, 16)
    _assert_close(got, _oracle(oracle_lib, inp, 16))


def test_paper_block_size_full_length_all_rows(tt, oracle_lib):
    # S = 16 (the final configuration of Section 2.3), 4096 tokens, 256 blocks
    B, N, S = 2, 4096, 16
    inp = _inputs(B, N, 32, 2, 128, seed=0)
    ref = _oracle(oracle_lib, inp, S)
    for sched in KERNELS:
        with attn_schedule(tt, *sched):
            got = _run_gpu(tt, inp, S)
        _assert_close(got, ref)


def test_invalid_block_size_raises(tt):
    import torch
    q = torch.zeros(1, 30, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 30, 1, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 1, 30, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tt.TTError):
        tt.block_attn_train(q, k, k, kc, kc, 7)
