"""GPU parity of tt_commit against the scalar CPU oracle, bit for bit.

Unmask/commit, "Nemotron-Labs-TwoTower" Section 2.2, Algorithm 2, with a fixed
budget of k commits per block per step. On identical fp32 logits the GPU and
the oracle must agree exactly on the canonical confidence keys, the greedy
predictions, the committed set (ascending-row tie-break) and the updated ids
and mask.
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


def _gpu_step(tt, logits, B, L, masked, k, tok, alias=False):
    import torch
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    m = torch.from_numpy(masked.copy()).cuda()
    t = torch.from_numpy(tok.copy()).cuda()
    mo = m if alias else None
    t, mo = tt.commit(lg, B, L, m, k, t, masked_out=mo)
    keys, args = tt.commit_keys(B * L)
    torch.cuda.synchronize()
    assert tt.handle().get_error() == 0
    return (t.cpu().numpy(), mo.cpu().numpy(), keys.cpu().numpy().view(np.uint64),
            args.cpu().numpy())


def _check_step(tt, oracle_lib, logits, B, L, masked, k, tok, alias=False):
    gt, gm, gk, ga = _gpu_step(tt, logits, B, L, masked, k, tok, alias)
    ot, om, ok, oa = oracle_lib.commit(logits, B, L, masked, k, tok)
    sel = masked == 1
    np.testing.assert_array_equal(gk[sel], ok[sel])
    np.testing.assert_array_equal(ga[sel], oa[sel])
    np.testing.assert_array_equal(gt, ot)
    np.testing.assert_array_equal(gm, om)
    return ot, om


def test_tiny_full_denoise_loop(tt, oracle_lib):
    w = wl.WORKLOADS["tiny_c256_l32"]
    tok = np.full(w.rows, -1, np.int32)
    masked = np.ones(w.rows, np.uint8)
    steps = 0
    while masked.any():
        lg = wl.logits(w, seed=0, step=steps)
        tok, masked = _check_step(tt, oracle_lib, lg, w.B, w.L, masked, w.k, tok)
        steps += 1
    assert steps == 8


@pytest.mark.parametrize("case", [
    # B, L, V, k, mask fraction
    (4, 32, 1024, 4, 1.0),
    (3, 50, 1000, 7, 0.6),      # V not a multiple of the cluster slice
    (2, 300, 4096, 64, 0.9),    # L above one warp per row group
    (5, 16, 2048, 1, 0.7),      # mock autoregressive mode: k = 1
    (2, 24, 512, 100, 0.5),     # k above #masked: commit all
    (1, 1, 4, 1, 1.0),          # smallest shape
    (2, 1030, 256, 9, 0.8),     # L above the select kernel's 1024 threads
    (2, 24, 100000, 5, 0.8),    # each CTA's quarter ends in a partial 16384-logit chunk
    (1, 16, 131068, 3, 1.0),    # largest V below the limit: the last quarter is ragged
    (1, 4100, 64, 37, 0.7),     # L above the 2048 staged keys: ranks counted chunk by chunk
    (2, 16384, 16, 300, 0.5),   # the largest block (16384 rows); V = 16 makes key ties common
    (4096, 4, 64, 1, 0.6),      # many small blocks: each cluster's share spans ~100 blocks
])
def test_shapes_and_masks(tt, oracle_lib, case):
    B, L, V, k, frac = case
    w = wl.custom("c", B, L, 1, 1, 8, 8, (0,) * B, V=V, k=k)
    lg = wl.logits(w, seed=11)
    masked = wl.random_mask(w, frac, seed=5) if frac < 1 else np.ones(w.rows, np.uint8)
    tok = np.arange(w.rows, dtype=np.int32) + 7
    _check_step(tt, oracle_lib, lg, B, L, masked, k, tok)


def test_argmax_in_partial_chunks_and_every_quarter(tt, oracle_lib):
    # V = 100000: quarters of 25000 logits, the second chunk of each holds
    # 8616. Plant each row's maximum in a different place: the last logit of
    # a quarter (inside its partial chunk), the first logit of a quarter, a
    # tie between two quarters (the lower id wins), and the last logit of the row.
    V = 100000
    w = wl.custom("plant", 2, 16, 1, 1, 8, 8, (0, 0), V=V, k=4)
    lg = wl.logits(w, seed=13)
    spots = [24999, 25000, 49999, 50000, 74999, 75000, 99999, 16383, 16384, 41383, 41384,
             0, 66383, 91384, 12345, 99996]
    for r, v in enumerate(spots):
        lg[r, v] = 30.0
    lg[16, [30000, 80000]] = 30.0    # tie across quarters -> 30000
    lg[17, [24999, 25000]] = 30.0    # tie across the quarter boundary -> 24999
    lg[18, :] = -2.0
    lg[18, 99999] = -1.0             # the maximum is the very last logit
    masked = np.ones(w.rows, np.uint8)
    tok = np.full(w.rows, -1, np.int32)
    _check_step(tt, oracle_lib, lg, 2, 16, masked, 4, tok)


def test_ties_and_alias(tt, oracle_lib):
    w = wl.custom("ties", 2, 40, 1, 1, 8, 8, (0, 0), V=2048, k=6)
    lg = wl.logits(w, seed=12)
    lg[3] = lg[10]                   # identical rows -> identical keys; row 3 first
    lg[50] = lg[41]
    lg[7, [100, 900]] = 40.0         # argmax tie -> lower vocab id
    lg[8] = 0.0                      # flat row
    lg[9, :] = -1e30
    lg[9, 5] = 3.0                   # confidence 1 (other terms underflow to 0)
    masked = np.ones(w.rows, np.uint8)
    masked[[0, 44]] = 0
    lg[0] = np.nan                   # unmasked rows are never read
    tok = np.full(w.rows, -1, np.int32)
    _check_step(tt, oracle_lib, lg, 2, 40, masked, 6, tok, alias=True)


@pytest.mark.parametrize("L,k", [(256, 1), (256, 8), (256, 95), (256, 96), (256, 97),
                                 (256, 128), (256, 200), (256, 229), (200, 7), (200, 150),
                                 (33, 20)])
def test_selection_budgets_and_key_ties(tt, oracle_lib, L, k):
    # Blocks of up to 256 rows: budgets up to 96 take the per-round warp
    # minimum, larger ones the binary search on the key. Identical logit rows
    # give identical keys in different lanes and in one lane (rows 8 apart
    # and adjacent), some of them at the cut of the budget; the lower row wins.
    w = wl.custom("sel", 2, L, 1, 1, 8, 8, (0, 0), V=2048, k=k)
    lg = wl.logits(w, seed=21)
    seen = set()
    groups = []
    for g in ([3, 11, 100, L - 1], [40, 41, 42, 43, 44], [7, 200, 129]):
        g = [r % L for r in g if r % L not in seen]
        seen.update(g)
        groups.append(g)
    for b in range(2):
        for g in groups:
            for r in g[1:]:
                lg[b * L + r] = lg[b * L + g[0]]
    masked = wl.random_mask(w, 0.9, seed=8)
    masked[[3, L + groups[1][0]]] = 1
    tok = np.full(w.rows, -1, np.int32)
    _check_step(tt, oracle_lib, lg, 2, L, masked, k, tok)


@pytest.mark.parametrize("rank", [0, 30, 120, 180])
def test_selection_cut_inside_a_key_tie(tt, oracle_lib, rank):
    # The row at confidence rank `rank` of block 0 is copied to four rows in
    # different lanes and one lane (rows 8 apart and adjacent); the budget
    # ends in the middle of that tie (the per-round path below 96 commits, the
    # binary search above), so the lower rows of the tie commit.
    L, V = 256, 2048
    w = wl.custom("cut", 2, L, 1, 1, 8, 8, (0, 0), V=V, k=1)
    lg = wl.logits(w, seed=23)
    masked = wl.random_mask(w, 0.9, seed=9)
    masked[:L][[5, 6, 13, 77, 160]] = 1
    _, _, keys, _ = oracle_lib.commit(lg, 2, L, masked, 1, np.full(w.rows, -1, np.int32))
    cand = [r for r in np.argsort(keys[:L], kind="stable") if masked[r] and r not in (5, 6, 13, 77, 160)]
    src = cand[rank]
    for r in (5, 6, 13, 77, 160):
        lg[r] = lg[src]
    k = rank + 3  # the tie spans ranks rank .. rank + 5 (with src): cut after three
    tok = np.full(w.rows, -1, np.int32)
    _, om = _check_step(tt, oracle_lib, lg, 2, L, masked, k, tok)
    tie = sorted([5, 6, 13, 77, 160, int(src)])
    committed = [r for r in tie if om[r] == 0]
    assert 0 < len(committed) < len(tie)
    assert committed == tie[:len(committed)]


@pytest.mark.parametrize("name", ["b8_c4096_l32", "b16_c1024_l256", "b4_gen8k_32x256",
                                  "b64_ragged8k32k_l64"])
def test_full_workloads_first_step(tt, oracle_lib, name):
    w = wl.WORKLOADS[name]
    inp = wl.commit_inputs(w, seed=0)
    _check_step(tt, oracle_lib, inp.logits, w.B, w.L, inp.masked, w.k, inp.tok)


@pytest.mark.parametrize("alias", [False, True], ids=["separate", "in_place"])
@pytest.mark.parametrize("name", ["b4_gen8k_32x256", "b64_ragged8k32k_l64"])
def test_full_workloads_ragged_mask(tt, oracle_lib, name, alias):
    # a later denoising step: about half of each block still masked, a different
    # set per block, so cluster shares start and end inside blocks and include
    # unmasked rows; in place, the mask is rewritten while other clusters run
    w = wl.WORKLOADS[name]
    lg = wl.logits(w, seed=0, step=3)
    masked = wl.random_mask(w, 0.5, seed=17)
    tok = np.where(masked == 1, -1, np.arange(w.rows) % w.V).astype(np.int32)
    _check_step(tt, oracle_lib, lg, w.B, w.L, masked, w.k, tok, alias=alias)


def test_canonical_key_at_reduction_boundaries(tt, oracle_lib):
    # Differences l - max at which rounding x*log2(e) to fp32 first would move
    # the exponential's n by one (the product is within half an fp32 ulp of a
    # half-integer): the keys must still agree with the oracle bit for bit.
    l2e = np.float32(1.0 / 0.69314718055994530942)
    xs = []
    for k in range(44):
        x0 = np.float32(-(k + 0.5) / float(l2e))
        for d in range(-40, 41):
            x = np.array([x0.view(np.int32) + d], np.int32).view(np.float32)[0]
            if -30.0 <= x <= 0.0:
                xs.append(x)
    xs = np.array(xs, np.float32)
    V = 4096
    rows = -(-len(xs) // (V - 1))
    w = wl.custom("bnd", 1, max(rows, 2), 1, 1, 8, 8, (0,), V=V, k=1)
    lg = wl.logits(w, seed=21) - np.float32(40.0)   # every other term is 0
    flat = lg.reshape(-1)
    for r in range(w.rows):
        lg[r, 0] = 0.0                                 # the row maximum
        chunk = xs[r * (V - 1):(r + 1) * (V - 1)]
        lg[r, 1:1 + len(chunk)] = chunk                # l - max = x exactly
    assert flat.size == w.rows * V
    masked = np.ones(w.rows, np.uint8)
    _check_step(tt, oracle_lib, lg, 1, w.rows, masked, 1, np.full(w.rows, -1, np.int32))


def test_b8_full_loop(tt, oracle_lib):
    w = wl.WORKLOADS["b8_c4096_l32"]
    tok = np.full(w.rows, -1, np.int32)
    masked = np.ones(w.rows, np.uint8)
    for step in range(w.steps_to_unmask):
        lg = wl.logits(w, seed=0, step=step)
        tok, masked = _check_step(tt, oracle_lib, lg, w.B, w.L, masked, w.k, tok)
    assert not masked.any()
