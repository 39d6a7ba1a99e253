"""Pins of the oracle's training-time batched block attention.

"Nemotron-Labs-TwoTower" Section 2.3, "Implementation": the denoiser processes
all noisy blocks of a clean sequence in one forward pass; its attention layers
attend to past clean context blocks and bidirectionally within the current
noisy block. The checks:

* against a library routine: torch scaled_dot_product_attention in float64 over
  the whole sequence at once, keys [clean tokens; noisy tokens] with the
  block-diagonal + clean-prefix boolean mask;
* one block (N = S) -> plain bidirectional attention over the block;
* noisy block j never reads clean positions at or past j*S (poisoned with NaN
  they change nothing), and block 0 reads no clean position at all;
* rows mode equals the full output.
"""
import numpy as np
import pytest
import torch

from block_diffusion_decoding_attn_b300 import workload as wl

TOL = 1e-10


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _inputs(B, N, Hq, Hkv, D, seed):
    # q [B][N][Hq][D]; k_blk/v_blk [B][N][Hkv][D] are the noisy tokens;
    # k_ctx/v_ctx [B][Hkv][N][D] the clean ones
    w = wl.custom("train", B, N, Hq, Hkv, D, N, (N,) * B, qk_std=1.0)
    return wl.attn_inputs(w, seed=seed)


def _train(o, inp, S, **kw):
    return o.block_attn_train(inp.q, inp.k_blk, inp.v_blk, inp.k_ctx, inp.v_ctx, S, **kw)


def _dense_masked_sdpa(inp, S):
    B, N, Hq, D = inp.q.shape
    Hkv = inp.k_ctx.shape[1]
    G = Hq // Hkv
    pos = np.arange(N)
    blk = pos // S
    # query n sees clean key c iff c < blk(n)*S, noisy key m iff blk(m) == blk(n)
    clean_ok = pos[None, :] < (blk * S)[:, None]
    noisy_ok = blk[None, :] == blk[:, None]
    mask = torch.from_numpy(np.concatenate([clean_ok, noisy_ok], axis=1))  # [N][2N]
    outs = []
    for b in range(B):
        k = np.concatenate([_f64(inp.k_ctx[b]), _f64(inp.k_blk[b]).transpose(1, 0, 2)], 1)
        v = np.concatenate([_f64(inp.v_ctx[b]), _f64(inp.v_blk[b]).transpose(1, 0, 2)], 1)
        k = torch.from_numpy(k).repeat_interleave(G, dim=0)
        v = torch.from_numpy(v).repeat_interleave(G, dim=0)
        q = torch.from_numpy(_f64(inp.q[b]).transpose(1, 0, 2).copy())
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=inp.scale)
        outs.append(o.numpy().transpose(1, 0, 2))
    return np.stack(outs)


CASES = [
    # name, B, N, S, Hq, Hkv, D
    ("s4_gqa2", 2, 12, 4, 4, 2, 8),
    ("s3_mha", 1, 9, 3, 3, 3, 16),
    ("s8_gqa8", 2, 24, 8, 8, 1, 32),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_dense_masked_sdpa(oracle_lib, case):
    name, B, N, S, Hq, Hkv, D = case
    inp = _inputs(B, N, Hq, Hkv, D, seed=21)
    np.testing.assert_allclose(_train(oracle_lib, inp, S), _dense_masked_sdpa(inp, S), rtol=0,
                               atol=TOL)


def test_one_block_is_bidirectional_attention(oracle_lib):
    inp = _inputs(2, 6, 4, 2, 8, seed=3)
    got = _train(oracle_lib, inp, 6)
    for b in range(2):
        q = torch.from_numpy(_f64(inp.q[b]).transpose(1, 0, 2).copy())
        k = torch.from_numpy(_f64(inp.k_blk[b]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
        v = torch.from_numpy(_f64(inp.v_blk[b]).transpose(1, 0, 2).copy()).repeat_interleave(2, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=inp.scale)
        np.testing.assert_allclose(got[b], ref.numpy().transpose(1, 0, 2), rtol=0, atol=TOL)


def test_block_reads_only_the_clean_prefix(oracle_lib):
    B, N, S = 2, 20, 5
    inp = _inputs(B, N, 4, 1, 8, seed=8)
    ref = _train(oracle_lib, inp, S)
    nan = np.uint16(0x7FC0)
    for j in range(N // S):
        k_save, v_save = inp.k_ctx.copy(), inp.v_ctx.copy()
        inp.k_ctx[:, :, j * S:, :] = nan
        inp.v_ctx[:, :, j * S:, :] = nan
        got = _train(oracle_lib, inp, S)
        sl = slice(j * S, (j + 1) * S)
        np.testing.assert_array_equal(got[:, sl], ref[:, sl])
        inp.k_ctx[...], inp.v_ctx[...] = k_save, v_save
    # and the clean prefix does matter for every later block
    inp.v_ctx[...] = 0
    got = _train(oracle_lib, inp, S)
    np.testing.assert_array_equal(got[:, :S], ref[:, :S])
    assert np.abs(got[:, S:] - ref[:, S:]).max() > 1e-3


def test_rows_mode_and_bad_block_size(oracle_lib):
    inp = _inputs(2, 16, 4, 2, 8, seed=5)
    full = _train(oracle_lib, inp, 4)
    rows = np.array([[0, 0, 0], [1, 15, 3], [0, 7, 2], [1, 8, 1], [1, 4, 0]], np.int32)
    part = _train(oracle_lib, inp, 4, rows=rows)
    for i, (b, n, h) in enumerate(rows):
        np.testing.assert_array_equal(part[i], full[b, n, h])
    with pytest.raises(ValueError):
        _train(oracle_lib, inp, 5)
