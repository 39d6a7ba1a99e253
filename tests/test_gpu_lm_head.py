"""GPU parity of the LM head and the commit behind it (tt_lm_head,
tt_commit_rowmax) against the CPU oracle.

The LM head is the denoiser's output layer that Section 2.2's sampling
(Algorithm 2) reads: logits = hidden @ weight^T, bf16 inputs, fp32
accumulation. Tolerance on N(0, 1) inputs: each logit is a sum of K exact
bf16 products accumulated in fp32; K * 2^-23 of the largest |logit| bounds the
accumulation error whatever the rounding of each add (3.2e-4 at K = 2688), so
the test allows max|gpu - oracle| <= K * 2^-23 * max|oracle|.

The commit behind it is checked end to end from the seeded inputs alone. On
integer-valued inputs (lm_head_exact_inputs) every partial sum is exact in
fp32, so the tensor-core logits must equal the oracle's fp64 logits bit for
bit, and the GPU's commit (tt_commit_rowmax, and tt_commit on the same
logits) must equal the oracle's commit on the oracle's own logits bit for bit
(acceptance: bit-exact on identical fp32 logits). Small integers make tied
maxima and tied confidences common, so the first-argmax and row-order rules
are exercised too.
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


def _exact_ref(oracle_lib, hid, w, rows=None):
    """The oracle's logits of integer-valued inputs, as the fp32 values they are."""
    ref = oracle_lib.lm_head(hid, w, rows=rows)
    r32 = ref.astype(np.float32)
    assert np.array_equal(r32.astype(np.float64), ref), "inputs are not exact in fp32"
    return r32


@pytest.mark.parametrize("M,K,V", [(1, 8, 4), (130, 64, 260), (256, 136, 1024), (200, 2688, 4100),
                                   (129, 512, 513 * 4)])
def test_logits_exact_on_integer_inputs(tt, oracle_lib, M, K, V):
    hid, w = wl.lm_head_exact_inputs(M, K, V, seed=M + K)
    np.testing.assert_array_equal(_logits(tt, hid, w).cpu().numpy(), _exact_ref(oracle_lib, hid, w))


def _block_rows(L, blocks):
    return np.concatenate([np.arange(b * L, (b + 1) * L) for b in blocks])


def _commit_pair(tt, oracle_lib, hid, wt, B, L, masked, k, tok, alias, blocks=None):
    """GPU: tt_lm_head, then tt_commit_rowmax on its logits, and tt_commit on
    the same logits. Oracle: its own LM head, then its commit, on the rows of
    `blocks` (every block if None). Bit for bit: logits, keys, predictions,
    tokens and mask. Returns the GPU's tokens and mask (numpy)."""
    import torch
    blocks = list(range(B)) if blocks is None else list(blocks)
    rows = _block_rows(L, blocks)
    lg = _logits(tt, hid, wt)
    ref = _exact_ref(oracle_lib, hid, wt, rows=None if len(blocks) == B else rows)
    rows_t = torch.from_numpy(rows).cuda()
    np.testing.assert_array_equal(lg.index_select(0, rows_t).cpu().numpy(), ref)
    m = torch.from_numpy(masked.copy()).cuda()
    t = torch.from_numpy(tok.copy()).cuda()
    mo = m if alias else torch.empty_like(m)
    tt.commit_rowmax(lg, B, L, m, k, t, masked_out=mo)
    keys, args = tt.commit_keys(B * L)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    got_t, got_m = t.cpu().numpy(), mo.cpu().numpy()
    ot, om, ok, oa = oracle_lib.commit(ref, len(blocks), L, masked[rows], k, tok[rows])
    sel = masked[rows] == 1
    np.testing.assert_array_equal(keys.cpu().numpy().view(np.uint64)[rows][sel], ok[sel])
    np.testing.assert_array_equal(args.cpu().numpy()[rows][sel], oa[sel])
    np.testing.assert_array_equal(got_t[rows], ot)
    np.testing.assert_array_equal(got_m[rows], om)
    # the cluster commit on the same logits: the same result on every row
    m2 = torch.from_numpy(masked.copy()).cuda()
    t2 = torch.from_numpy(tok.copy()).cuda()
    t2, mo2 = tt.commit(lg, B, L, m2, k, t2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t2.cpu().numpy(), got_t)
    np.testing.assert_array_equal(mo2.cpu().numpy(), got_m)
    # every block: min(k, #masked) rows commit, only masked rows change
    n_in = masked.reshape(B, L).astype(np.int64).sum(1)
    n_out = got_m.reshape(B, L).astype(np.int64).sum(1)
    np.testing.assert_array_equal(n_in - n_out, np.minimum(k, n_in))
    assert not got_m[masked == 0].any()
    np.testing.assert_array_equal(got_t[masked == 0], tok[masked == 0])
    return got_t, got_m


@pytest.mark.parametrize("alias", [False, True], ids=["separate", "in_place"])
@pytest.mark.parametrize("B,L,K,V,k,frac", [(4, 32, 256, 4096, 4, 1.0), (3, 50, 136, 1000, 7, 0.6),
                                            (2, 300, 64, 8200, 64, 0.9), (1, 1, 8, 4, 1, 1.0),
                                            (1, 4100, 8, 64, 37, 0.7), (1, 16384, 8, 64, 300, 0.5),
                                            (4096, 4, 8, 64, 1, 0.6)])
def test_commit_behind_the_lm_head(tt, oracle_lib, B, L, K, V, k, frac, alias):
    w = wl.custom("lmc", B, L, 1, 1, 8, 8, (0,) * B, V=V, k=k)
    hid, wt = wl.lm_head_exact_inputs(B * L, K, V, seed=7 + L)
    masked = wl.random_mask(w, frac, seed=3) if frac < 1 else np.ones(w.rows, np.uint8)
    tok = np.arange(w.rows, dtype=np.int32) + 5
    _commit_pair(tt, oracle_lib, hid, wt, B, L, masked, k, tok, alias)


def test_denoise_loop_with_fresh_hidden_states(tt, oracle_lib):
    # every step: a new hidden state through the LM head, then the commit in place
    B, L, K, V, k = 4, 64, 256, 8192, 8
    tok = np.full(B * L, -1, np.int32)
    masked = np.ones(B * L, np.uint8)
    _, wt = wl.lm_head_exact_inputs(1, K, V, seed=11)
    for step in range(L // k):
        hid, _ = wl.lm_head_exact_inputs(B * L, K, V, seed=11, step=step)
        tok, masked = _commit_pair(tt, oracle_lib, hid, wt, B, L, masked, k, tok, alias=True)
    assert not masked.any()
    assert (tok >= 0).all() and (tok < V).all()


def test_full_size_ragged_workload_shapes(tt, oracle_lib):
    # b64_ragged8k32k_l64's commit shape (4096 rows, V = 131072) at the pages'
    # width K = 2688: sampled logit rows of N(0, 1) inputs against the oracle
    # within the tolerance; then, on integer-valued inputs, the logits and the
    # whole commit of three sampled blocks bit for bit against the oracle's,
    # and the per-block commit counts on every block
    w = wl.WORKLOADS["b64_ragged8k32k_l64"]
    K = wl.LM_HIDDEN
    hid, wt = wl.lm_head_inputs(w.rows, K, w.V, seed=0)
    lg = _logits(tt, hid, wt)
    rows = [0, 1, 777, 2048, 4095]
    ref = oracle_lib.lm_head(hid, wt, rows=rows)
    got = lg[rows].cpu().numpy().astype(np.float64)
    assert np.abs(got - ref).max() <= K * 2.0 ** -23 * np.abs(ref).max()
    del lg
    hid, wt = wl.lm_head_exact_inputs(w.rows, K, w.V, seed=0)
    masked = wl.random_mask(w, 0.5, seed=21)
    tok = np.full(w.rows, -1, np.int32)
    _commit_pair(tt, oracle_lib, hid, wt, w.B, w.L, masked, w.k, tok, alias=True,
                 blocks=[0, 37, w.B - 1])


def test_shape_mismatch_is_rejected(tt):
    import torch
    hid, wt = wl.lm_head_inputs(64, 64, 256, seed=1)
    lg = _logits(tt, hid, wt)
    m = torch.ones(32, dtype=torch.uint8, device="cuda")
    t = torch.zeros(32, dtype=torch.int32, device="cuda")
    with pytest.raises(tt.TTError):
        tt.commit_rowmax(lg[:32].contiguous(), 1, 32, m, 1, t)
