"""Pins of the CPU attention oracle against what the pages and mathematics fix.

"Nemotron-Labs-TwoTower" Section 2.1, Eq. (1): queries of the noisy block take
one softmax over [context-tower keys of the layer; the block's own keys], with
no mask inside the block and causality to past clean blocks. The checks:

* the general case against a library routine (torch scaled_dot_product_attention
  in float64 on the explicitly concatenated, GQA-expanded key list);
* empty context -> plain bidirectional attention over the block;
* block of one -> the last row of causal attention over [context; token];
* invariants: block-token permutation equivariance, context permutation
  invariance, constant values, zero scale gives the mean of the values;
* brute force with Python's math module on a tiny case;
* positions at or past ctx_len are never read (they hold NaN).
"""
import math

import numpy as np
import pytest
import torch

from block_diffusion_decoding_attn_b300 import workload as wl

TOL = 1e-10


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _sdpa_reference(inp, causal_last=False):
    """Eq. (1) through torch SDPA (float64), one sequence at a time."""
    B, L, Hq, D = inp.q.shape
    Hkv = inp.k_ctx.shape[1]
    G = Hq // Hkv
    outs = []
    for b in range(B):
        C = int(inp.ctx_len[b])
        k = np.concatenate([_f64(inp.k_ctx[b, :, :C, :]), _f64(inp.k_blk[b]).transpose(1, 0, 2)], 1)
        v = np.concatenate([_f64(inp.v_ctx[b, :, :C, :]), _f64(inp.v_blk[b]).transpose(1, 0, 2)], 1)
        k = torch.from_numpy(k).repeat_interleave(G, dim=0)  # [Hq][N][D]
        v = torch.from_numpy(v).repeat_interleave(G, dim=0)
        q = torch.from_numpy(_f64(inp.q[b]).transpose(1, 0, 2).copy())  # [Hq][L][D]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=inp.scale)
        outs.append(o.numpy().transpose(1, 0, 2))
    return np.stack(outs)


CASES = [
    # name, B, L, Hq, Hkv, D, cap, ctx
    ("gqa4_ragged", 2, 7, 8, 2, 16, 40, (13, 40)),
    ("mha", 1, 5, 3, 3, 8, 9, (9,)),
    ("gqa16_d64", 2, 4, 16, 1, 64, 33, (0, 21)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_general_case_matches_sdpa(oracle_lib, case):
    name, B, L, Hq, Hkv, D, cap, ctx = case
    w = wl.custom(name, B, L, Hq, Hkv, D, cap, ctx, qk_std=1.0)
    inp = wl.attn_inputs(w, seed=3)
    got = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    ref = _sdpa_reference(inp)
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL)


def test_empty_context_is_bidirectional_attention(oracle_lib):
    w = wl.custom("empty", 1, 6, 4, 2, 8, 4, (0,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=5)
    got = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    q = torch.from_numpy(_f64(inp.q[0]).transpose(1, 0, 2).copy())
    k = torch.from_numpy(_f64(inp.k_blk[0]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
    v = torch.from_numpy(_f64(inp.v_blk[0]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=False,
                                                           scale=inp.scale)
    np.testing.assert_allclose(got[0], ref.numpy().transpose(1, 0, 2), rtol=0, atol=TOL)
    # and it is not causal: the first query sees later block tokens
    causal = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                              scale=inp.scale)
    assert np.abs(got[0][0] - causal.numpy().transpose(1, 0, 2)[0]).max() > 1e-3


def test_block_of_one_is_causal_decode(oracle_lib):
    C, Hq, Hkv, D = 11, 4, 1, 16
    w = wl.custom("l1", 1, 1, Hq, Hkv, D, 16, (C,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=7)
    got = oracle_lib.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len)
    rng = np.random.default_rng(0)
    qs = np.concatenate([rng.standard_normal((Hq, C, D)), _f64(inp.q[0]).transpose(1, 0, 2)], 1)
    ks = np.concatenate([_f64(inp.k_ctx[0, :, :C]), _f64(inp.k_blk[0]).transpose(1, 0, 2)], 1)
    vs = np.concatenate([_f64(inp.v_ctx[0, :, :C]), _f64(inp.v_blk[0]).transpose(1, 0, 2)], 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qs), torch.from_numpy(ks).repeat_interleave(Hq, 0),
        torch.from_numpy(vs).repeat_interleave(Hq, 0), is_causal=True, scale=inp.scale)
    np.testing.assert_allclose(got[0, 0], ref.numpy()[:, -1, :], rtol=0, atol=TOL)


def _run(o, inp, **kw):
    return o.block_attn(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, inp.ctx_len, **kw)


def test_permuting_block_tokens_permutes_outputs(oracle_lib):
    w = wl.custom("perm", 1, 9, 4, 2, 16, 20, (17,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=11)
    base = _run(oracle_lib, inp)
    perm = np.random.default_rng(1).permutation(9)
    inp.q, inp.k_blk, inp.v_blk = inp.q[:, perm], inp.k_blk[:, perm], inp.v_blk[:, perm]
    np.testing.assert_allclose(_run(oracle_lib, inp), base[:, perm], rtol=0, atol=TOL)


def test_permuting_context_leaves_output_unchanged(oracle_lib):
    w = wl.custom("cperm", 1, 5, 4, 2, 16, 20, (20,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=13)
    base = _run(oracle_lib, inp)
    perm = np.random.default_rng(2).permutation(20)
    inp.k_ctx, inp.v_ctx = inp.k_ctx[:, :, perm], inp.v_ctx[:, :, perm]
    np.testing.assert_allclose(_run(oracle_lib, inp), base, rtol=0, atol=TOL)


def test_constant_values_and_zero_scale(oracle_lib):
    w = wl.custom("const", 2, 6, 4, 2, 8, 12, (12, 3), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=17)
    c = wl.to_bf16_bits(np.arange(8, dtype=np.float32) * 0.25 - 1.0)
    inp.v_ctx[:] = c
    inp.v_blk[:] = c
    out = _run(oracle_lib, inp)
    np.testing.assert_allclose(out, np.broadcast_to(_f64(c), out.shape), rtol=0, atol=TOL)
    # scale 0: uniform weights -> mean of the C_b + L values
    inp = wl.attn_inputs(w, seed=19)
    out = _run(oracle_lib, inp, scale=0.0)
    for b in range(2):
        C = int(inp.ctx_len[b])
        for h in range(4):
            kv = h // 2
            vals = np.concatenate([_f64(inp.v_ctx[b, kv, :C]), _f64(inp.v_blk[b, :, kv])])
            np.testing.assert_allclose(out[b, :, h], np.broadcast_to(vals.mean(0), (6, 8)),
                                       rtol=0, atol=TOL)


def test_brute_force_tiny(oracle_lib):
    w = wl.custom("tiny_bf", 1, 3, 2, 1, 4, 5, (4,), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=23)
    got = _run(oracle_lib, inp)
    q, kb, vb = _f64(inp.q), _f64(inp.k_blk), _f64(inp.v_blk)
    kc, vc = _f64(inp.k_ctx), _f64(inp.v_ctx)
    for l in range(3):
        for h in range(2):
            keys = [kc[0, 0, j] for j in range(4)] + [kb[0, j, 0] for j in range(3)]
            vals = [vc[0, 0, j] for j in range(4)] + [vb[0, j, 0] for j in range(3)]
            s = [sum(q[0, l, h, d] * kk[d] for d in range(4)) * 0.5 for kk in keys]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            ref = [sum(e[j] * vals[j][d] for j in range(7)) / z for d in range(4)]
            np.testing.assert_allclose(got[0, l, h], ref, rtol=0, atol=1e-12)


def test_padding_is_never_read_and_rows_mode(oracle_lib):
    w = wl.custom("pad", 2, 4, 4, 2, 16, 64, (5, 0), qk_std=1.0)
    inp = wl.attn_inputs(w, seed=29)  # positions >= ctx_len hold NaN
    full = _run(oracle_lib, inp)
    assert np.isfinite(full).all()
    rows = np.array([[1, 3, 2], [0, 0, 0], [0, 2, 3]], np.int32)
    part = _run(oracle_lib, inp, rows=rows)
    for i, (b, l, h) in enumerate(rows):
        np.testing.assert_array_equal(part[i], full[b, l, h])


def test_invalid_arguments_raise(oracle_lib):
    w = wl.custom("bad", 1, 2, 4, 2, 8, 4, (4,))
    inp = wl.attn_inputs(w, seed=1)
    inp.ctx_len = np.array([5], np.int32)  # beyond the cache capacity
    with pytest.raises(ValueError):
        _run(oracle_lib, inp)
