"""GPU parity of tt_commit_threshold against the scalar CPU oracle, bit for bit.

"Nemotron-Labs-TwoTower" Section 2.2, Algorithm 2 with a confidence threshold
gamma: per block, every masked row whose confidence (2^40 / key) is above gamma
commits, and at least ceil(#masked / steps_left). On identical fp32 logits the
GPU and the oracle must agree exactly on keys, predictions, committed sets,
ids and masks.
"""
import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tt():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_diffusion_decoding_attn_b300 as tt
    from block_diffusion_decoding_attn_b300 import build
    build.build()
    return tt


def _check(tt, oracle_lib, logits, B, L, masked, gamma, steps_left, tok):
    import torch
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    m = torch.from_numpy(masked.copy()).cuda()
    t = torch.from_numpy(tok.copy()).cuda()
    t, mo = tt.commit_threshold(lg, B, L, m, gamma, steps_left, t)
    gk, ga = tt.commit_keys(B * L)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    gk, ga = gk.cpu().numpy().view(np.uint64), ga.cpu().numpy()
    ot, om, ok, oa = oracle_lib.commit_threshold(logits, B, L, masked, gamma, steps_left, tok)
    sel = masked == 1
    np.testing.assert_array_equal(gk[sel], ok[sel])
    np.testing.assert_array_equal(ga[sel], oa[sel])
    np.testing.assert_array_equal(t.cpu().numpy(), ot)
    np.testing.assert_array_equal(mo.cpu().numpy(), om)
    return ot, om, ok


@pytest.mark.parametrize("case", [
    # B, L, V, mask fraction, steps_left
    (4, 32, 1024, 1.0, 8),
    (3, 50, 1000, 0.6, 3),
    (2, 300, 4096, 0.9, 5),     # L above the register select (general path)
    (5, 16, 2048, 0.7, 1),      # last step: everything commits
    (1, 1, 4, 1.0, 2),
    (1, 4100, 64, 0.8, 7),      # L above the 2048 staged keys: ranks counted chunk by chunk
])
@pytest.mark.parametrize("where", ["none", "median", "all"])
def test_threshold_shapes(tt, oracle_lib, case, where):
    B, L, V, frac, steps_left = case
    w = wl.custom("thr", B, L, 1, 1, 8, 8, (0,) * B, V=V, k=1, logit_std=3.0)
    lg = wl.logits(w, seed=31)
    masked = wl.random_mask(w, frac, seed=6) if frac < 1 else np.ones(w.rows, np.uint8)
    tok = np.arange(w.rows, dtype=np.int32) + 3
    if where == "none":
        gamma = 1.5
    elif where == "all":
        gamma = 0.0
    else:  # a gamma inside the confidence distribution, and exactly on one row's confidence
        _, _, keys, _ = oracle_lib.commit(lg, B, L, masked, 1, tok)
        conf = (1 << 40) / keys[masked == 1].astype(np.float64)
        gamma = float(np.median(conf))
    _check(tt, oracle_lib, lg, B, L, masked, gamma, steps_left, tok)


def test_threshold_denoise_loop(tt, oracle_lib):
    # gamma = 0.8 (the paper's sampling threshold), T = 8 steps on the small workload
    w = wl.WORKLOADS["tiny_c256_l32"]
    T = 8
    tok = np.full(w.rows, -1, np.int32)
    masked = np.ones(w.rows, np.uint8)
    for r in range(1, T + 1):
        lg = wl.logits(w, seed=0, step=r)
        tok, masked, _ = _check(tt, oracle_lib, lg, w.B, w.L, masked, 0.8, T - r + 1, tok)
    assert not masked.any()


def test_threshold_full_workload_first_step(tt, oracle_lib):
    w = wl.WORKLOADS["b8_c4096_l32"]
    inp = wl.commit_inputs(w, seed=0)
    _check(tt, oracle_lib, inp.logits, w.B, w.L, inp.masked, 0.02, 8, inp.tok)
