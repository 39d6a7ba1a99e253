"""Pins of the oracle's context-tower update: causal block attention and K/V append.

"Nemotron-Labs-TwoTower" Section 2.1, Algorithm 1 (the context update after a commit):
once a block is clean the context tower runs its tokens causally over the prefix
cache, and the block's keys/values join that cache. The checks:

* causal attention against a library routine: torch scaled_dot_product_attention
  in float64 on the concatenated [context; block] list with an explicit boolean
  mask (query l sees the context and block keys 0..l);
* empty context -> SDPA with is_causal=True over the block alone;
* closed form: equal keys give the mean of the visible values, C + l + 1 of them;
* composition with the append and the (separately pinned) bidirectional oracle:
  causal row l equals a one-token block over the cache with block rows 0..l-1
  appended; block of one and last row equal the bidirectional result;
* the append against hand-written expected arrays, including a block that does
  not fit, and its invariants (rows outside the appended range unchanged).
"""
import numpy as np
import pytest
import torch

from block_diffusion_decoding_attn_b300 import workload as wl

TOL = 1e-10


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _sdpa_causal(inp):
    """The causal variant through torch SDPA (float64) with an explicit mask."""
    B, L, Hq, D = inp.q.shape
    Hkv = inp.k_ctx.shape[1]
    G = Hq // Hkv
    outs = []
    for b in range(B):
        C = int(inp.ctx_len[b])
        k = np.concatenate([_f64(inp.k_ctx[b, :, :C, :]), _f64(inp.k_blk[b]).transpose(1, 0, 2)], 1)
        v = np.concatenate([_f64(inp.v_ctx[b, :, :C, :]), _f64(inp.v_blk[b]).transpose(1, 0, 2)], 1)
        k = torch.from_numpy(k).repeat_interleave(G, dim=0)  # [Hq][C+L][D]
        v = torch.from_numpy(v).repeat_interleave(G, dim=0)
        q = torch.from_numpy(_f64(inp.q[b]).transpose(1, 0, 2).copy())  # [Hq][L][D]
        allowed = torch.arange(C + L)[None, :] <= (C + torch.arange(L))[:, None]  # [L][C+L]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed,
                                                             scale=inp.scale)
        outs.append(o.numpy().transpose(1, 0, 2))
    return np.stack(outs)


def _causal(o, inp, **kw):
    return o.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len,
                        causal=True, **kw)


CASES = [
    # name, B, L, Hq, Hkv, D, cap, ctx
    ("gqa4_ragged", 2, 7, 8, 2, 16, 40, (13, 40)),
    ("mha", 1, 5, 3, 3, 8, 9, (9,)),
    ("gqa16_d64", 2, 4, 16, 1, 64, 33, (0, 21)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_causal_matches_masked_sdpa(oracle_lib, case):
    name, B, L, Hq, Hkv, D, cap, ctx = case
    w = wl.custom(name, B, L, Hq, Hkv, D, cap, ctx, qk_std=1.0)
    inp = wl.attn_inputs(w, seed=11)
    np.testing.assert_allclose(_causal(oracle_lib, inp), _sdpa_causal(inp), rtol=0, atol=TOL)


def test_empty_context_is_causal_sdpa(oracle_lib):
    w = wl.custom("empty", 1, 6, 4, 2, 8, 4, (0,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=5)
    got = _causal(oracle_lib, inp)
    q = torch.from_numpy(_f64(inp.q[0]).transpose(1, 0, 2).copy())
    k = torch.from_numpy(_f64(inp.k_blk[0]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
    v = torch.from_numpy(_f64(inp.v_blk[0]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=inp.scale)
    np.testing.assert_allclose(got[0], ref.numpy().transpose(1, 0, 2), rtol=0, atol=TOL)


def test_equal_keys_average_the_visible_values(oracle_lib):
    # All keys zero: every visible key has score 0, so row l is the plain mean of
    # the C + l + 1 values it sees (a dropped or extra key changes the mean).
    w = wl.custom("eqk", 2, 5, 4, 2, 8, 12, (3, 0), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=2)
    inp.k_blk[...] = 0
    inp.k_ctx[...] = 0
    got = _causal(oracle_lib, inp)
    G = 2
    for b in range(2):
        C = int(inp.ctx_len[b])
        for l in range(5):
            for h in range(4):
                kv = h // G
                vis = np.concatenate([_f64(inp.v_ctx[b, kv, :C, :]), _f64(inp.v_blk[b, :l + 1, kv, :])])
                assert vis.shape[0] == C + l + 1
                np.testing.assert_allclose(got[b, l, h], vis.mean(axis=0), rtol=0, atol=1e-12)


def test_causal_row_is_decode_over_the_appended_cache(oracle_lib):
    # Row l of the causal pass = a one-token block (token l) attending over the
    # cache after block rows 0..l-1 were appended: ties the causal cut to the
    # bidirectional oracle and the append.
    w = wl.custom("compose", 2, 6, 8, 2, 16, 24, (5, 11), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=7)
    got = _causal(oracle_lib, inp)
    for l in range(6):
        kc, vc, n, fits = oracle_lib.kv_append(inp.k_blk[:, :l], inp.v_blk[:, :l], inp.k_ctx,
                                               inp.v_ctx, inp.ctx_len) if l else \
            (inp.k_ctx, inp.v_ctx, inp.ctx_len, np.ones(2, bool))
        assert fits.all()
        one = oracle_lib.block_attn(inp.q[:, l:l + 1], inp.k_blk[:, l:l + 1], inp.v_blk[:, l:l + 1],
                                    kc, vc, n)
        np.testing.assert_allclose(got[:, l], one[:, 0], rtol=0, atol=TOL)


def test_block_of_one_and_last_row_equal_bidirectional(oracle_lib):
    w = wl.custom("last", 2, 5, 4, 1, 8, 10, (10, 3), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=9)
    bi = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    ca = _causal(oracle_lib, inp)
    np.testing.assert_array_equal(ca[:, -1], bi[:, -1])
    assert np.abs(ca[:, 0] - bi[:, 0]).max() > 1e-3  # the first query no longer sees later tokens
    one = wl.custom("one", 2, 1, 4, 1, 8, 10, (10, 3), qk_std=1.0)
    inp1 = wl.attn_inputs(one, seed=9)
    np.testing.assert_array_equal(
        _causal(oracle_lib, inp1),
        oracle_lib.block_attn(inp1.q, inp1.k_blk, inp1.v_blk, inp1.k_ctx, inp1.v_ctx, inp1.ctx_len))


def test_causal_never_reads_cache_padding_and_rows_mode(oracle_lib):
    w = wl.custom("pad", 2, 4, 4, 2, 8, 16, (6, 0), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=4)
    nan = np.uint16(0x7FC0)
    inp.k_ctx[0, :, 6:, :] = nan
    inp.v_ctx[0, :, 6:, :] = nan
    inp.k_ctx[1] = nan
    inp.v_ctx[1] = nan
    full = _causal(oracle_lib, inp)
    assert np.isfinite(full).all()
    rows = np.array([[1, 3, 2], [0, 0, 1], [0, 2, 3]], np.int32)
    part = _causal(oracle_lib, inp, rows=rows)
    for i, (b, l, h) in enumerate(rows):
        np.testing.assert_array_equal(part[i], full[b, l, h])


def test_append_hand_written():
    # B=3, L=2, Hkv=2, D=2, cap=4. Sequence 0 has 1 cached row, sequence 1 has 3
    # (the block does not fit: unchanged), sequence 2 has 2 (fills the cache).
    from oracle import kv_append
    k_blk = np.array([[[[1, 2], [3, 4]], [[5, 6], [7, 8]]],
                      [[[9, 9], [9, 9]], [[9, 9], [9, 9]]],
                      [[[11, 12], [13, 14]], [[15, 16], [17, 18]]]], np.uint16)  # [b][l][h][d]
    v_blk = k_blk + 100
    k_ctx = np.full((3, 2, 4, 2), 0, np.uint16)  # fill values no block entry takes
    v_ctx = np.full((3, 2, 4, 2), 50, np.uint16)
    ctx_len = np.array([1, 3, 2], np.int32)
    kc, vc, n, fits = kv_append(k_blk, v_blk, k_ctx, v_ctx, ctx_len)
    expect_k = np.array([
        [[[0, 0], [1, 2], [5, 6], [0, 0]], [[0, 0], [3, 4], [7, 8], [0, 0]]],
        [[[0, 0], [0, 0], [0, 0], [0, 0]], [[0, 0], [0, 0], [0, 0], [0, 0]]],
        [[[0, 0], [0, 0], [11, 12], [15, 16]], [[0, 0], [0, 0], [13, 14], [17, 18]]],
    ], np.uint16)  # [b][h][pos][d]
    expect_v = np.array([
        [[[50, 50], [101, 102], [105, 106], [50, 50]], [[50, 50], [103, 104], [107, 108], [50, 50]]],
        [[[50, 50], [50, 50], [50, 50], [50, 50]], [[50, 50], [50, 50], [50, 50], [50, 50]]],
        [[[50, 50], [50, 50], [111, 112], [115, 116]], [[50, 50], [50, 50], [113, 114], [117, 118]]],
    ], np.uint16)
    np.testing.assert_array_equal(kc, expect_k)
    np.testing.assert_array_equal(vc, expect_v)
    np.testing.assert_array_equal(n, [3, 3, 4])
    np.testing.assert_array_equal(fits, [True, False, True])
    # inputs untouched
    assert (k_ctx == 0).all() and (v_ctx == 50).all() and list(ctx_len) == [1, 3, 2]


def test_append_invariants_on_random_data():
    from oracle import kv_append
    rng = np.random.default_rng(0)
    B, L, Hkv, D, cap = 4, 5, 3, 8, 16
    k_blk = rng.integers(0, 2**16, (B, L, Hkv, D), dtype=np.uint16)
    v_blk = rng.integers(0, 2**16, (B, L, Hkv, D), dtype=np.uint16)
    k_ctx = rng.integers(0, 2**16, (B, Hkv, cap, D), dtype=np.uint16)
    v_ctx = rng.integers(0, 2**16, (B, Hkv, cap, D), dtype=np.uint16)
    ctx_len = np.array([0, 11, 12, -1], np.int32)  # 11 fits exactly, 12 and -1 do not
    kc, vc, n, fits = kv_append(k_blk, v_blk, k_ctx, v_ctx, ctx_len)
    np.testing.assert_array_equal(fits, [True, True, False, False])
    np.testing.assert_array_equal(n, [5, 16, 12, -1])
    for b in range(B):
        c = int(ctx_len[b])
        if fits[b]:
            np.testing.assert_array_equal(kc[b, :, c:c + L], k_blk[b].transpose(1, 0, 2))
            np.testing.assert_array_equal(vc[b, :, c:c + L], v_blk[b].transpose(1, 0, 2))
            keep = np.ones(cap, bool)
            keep[c:c + L] = False
        else:
            keep = np.ones(cap, bool)
        np.testing.assert_array_equal(kc[b, :, keep], k_ctx[b, :, keep])
        np.testing.assert_array_equal(vc[b, :, keep], v_ctx[b, :, keep])
