"""GPU parity of the LM head and the commit behind it (tt_lm_head,
tt_commit_rowmax) against the CPU oracle.

The LM head is the denoiser's output layer that Section 2.2's sampling
(Algorithm 2) reads: logits = hidden @ weight^T, bf16 inputs, fp32
accumulation. Tolerance: each logit is a sum of K exact bf16 products
accumulated in fp32; K * 2^-23 of the largest |logit| bounds the accumulation
error whatever the rounding of each add (3.2e-4 at K = 2688), so the test
allows max|gpu - oracle| <= K * 2^-23 * max|oracle|.

The commit behind it must be bit-identical to the oracle's commit on the very
logits the GPU produced (acceptance: bit-exact on identical fp32 logits), and
to tt_commit on them.
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


def _dev_bf16(a):
    import torch
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def _logits(tt, hid, w):
    import torch
    lg = tt.lm_head(_dev_bf16(hid), _dev_bf16(w))
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    return lg


@pytest.mark.parametrize("M,K,V", [(1, 8, 4), (130, 64, 260), (256, 136, 1024), (200, 2688, 4100),
                                   (129, 512, 513 * 4)])
def test_logits_against_oracle(tt, oracle_lib, M, K, V):
    hid, w = wl.lm_head_inputs(M, K, V, seed=M + K)
    got = _logits(tt, hid, w).cpu().numpy().astype(np.float64)
    ref = oracle_lib.lm_head(hid, w)
    err = np.abs(got - ref).max()
    assert err <= K * 2.0 ** -23 * np.abs(ref).max(), err


def _commit_pair(tt, oracle_lib, lg, B, L, masked, k, tok, alias):
    """tt_commit_rowmax on lm_head's logits against the oracle and tt_commit on
    the same fp32 logits, bit for bit (tok, mask, keys, predictions)."""
    import torch
    m = torch.from_numpy(masked.copy()).cuda()
    t = torch.from_numpy(tok.copy()).cuda()
    mo = m if alias else torch.empty_like(m)
    tt.commit_rowmax(lg, B, L, m, k, t, masked_out=mo)
    keys, args = tt.commit_keys(B * L)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    lg_host = lg.cpu().numpy()
    ot, om, ok, oa = oracle_lib.commit(lg_host, B, L, masked, k, tok)
    sel = masked == 1
    np.testing.assert_array_equal(keys.cpu().numpy().view(np.uint64)[sel], ok[sel])
    np.testing.assert_array_equal(args.cpu().numpy()[sel], oa[sel])
    np.testing.assert_array_equal(t.cpu().numpy(), ot)
    np.testing.assert_array_equal(mo.cpu().numpy(), om)
    # the cluster commit on the same logits
    m2 = torch.from_numpy(masked.copy()).cuda()
    t2 = torch.from_numpy(tok.copy()).cuda()
    t2, mo2 = tt.commit(lg, B, L, m2, k, t2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t2.cpu().numpy(), ot)
    np.testing.assert_array_equal(mo2.cpu().numpy(), om)
    return ot, om


@pytest.mark.parametrize("alias", [False, True], ids=["separate", "in_place"])
@pytest.mark.parametrize("B,L,K,V,k,frac", [(4, 32, 256, 4096, 4, 1.0), (3, 50, 136, 1000, 7, 0.6),
                                            (2, 300, 64, 8200, 64, 0.9), (1, 1, 8, 4, 1, 1.0)])
def test_commit_behind_the_lm_head(tt, oracle_lib, B, L, K, V, k, frac, alias):
    w = wl.custom("lmc", B, L, 1, 1, 8, 8, (0,) * B, V=V, k=k)
    hid, wt = wl.lm_head_inputs(B * L, K, V, seed=7 + L)
    lg = _logits(tt, hid, wt)
    masked = wl.random_mask(w, frac, seed=3) if frac < 1 else np.ones(w.rows, np.uint8)
    tok = np.arange(w.rows, dtype=np.int32) + 5
    _commit_pair(tt, oracle_lib, lg, B, L, masked, k, tok, alias)


def test_denoise_loop_with_fresh_hidden_states(tt, oracle_lib):
    # every step: a new hidden state through the LM head, then the commit in place
    B, L, K, V, k = 4, 64, 256, 8192, 8
    tok = np.full(B * L, -1, np.int32)
    masked = np.ones(B * L, np.uint8)
    _, wt = wl.lm_head_inputs(1, K, V, seed=11)
    for step in range(L // k):
        hid, _ = wl.lm_head_inputs(B * L, K, V, seed=11, step=step)
        lg = _logits(tt, hid, wt)
        tok, masked = _commit_pair(tt, oracle_lib, lg, B, L, masked, k, tok, alias=True)
    assert not masked.any()


def test_full_size_ragged_workload_shapes(tt, oracle_lib):
    # b64_ragged8k32k_l64's commit shape (4096 rows, V = 131072) at the pages'
    # width K = 2688: sampled logit rows against the oracle, the whole commit
    # step against the oracle on the GPU's logits
    w = wl.WORKLOADS["b64_ragged8k32k_l64"]
    K = wl.LM_HIDDEN
    hid, wt = wl.lm_head_inputs(w.rows, K, w.V, seed=0)
    lg = _logits(tt, hid, wt)
    rows = [0, 1, 777, 2048, 4095]
    ref = oracle_lib.lm_head(hid, wt, rows=rows)
    got = lg[rows].cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= K * 2.0 ** -23 * np.abs(ref).max()
    masked = wl.random_mask(w, 0.5, seed=21)
    tok = np.full(w.rows, -1, np.int32)
    _commit_pair(tt, oracle_lib, lg, w.B, w.L, masked, w.k, tok, alias=True)


def test_shape_mismatch_is_rejected(tt):
    import torch
    hid, wt = wl.lm_head_inputs(64, 64, 256, seed=1)
    lg = _logits(tt, hid, wt)
    m = torch.ones(32, dtype=torch.uint8, device="cuda")
    t = torch.zeros(32, dtype=torch.int32, device="cuda")
    with pytest.raises(tt.TTError):
        tt.commit_rowmax(lg[:32].contiguous(), 1, 32, m, 1, t)
