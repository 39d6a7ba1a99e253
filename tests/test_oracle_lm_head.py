"""Pins of the CPU oracle's LM head (the step before Section 2.2's sampling:
logits = hidden @ weight^T over bf16 values, float64).

* brute force with Python loops on a tiny case (sums of exact products);
* closed forms that fix the orientation: a one-hot hidden row picks a weight
  column, an all-ones weight gives the row sums of hidden;
* the bf16 widening is exact (round trip of the generator's rounding).
"""
import math

import numpy as np

from block_diffusion_decoding_attn_b300 import workload as wl


def test_brute_force(oracle_lib):
    hid, w = wl.lm_head_inputs(3, 8, 5, seed=2)
    got = oracle_lib.lm_head(hid, w)
    h = oracle_lib.bf16_to_f64(hid)
    ww = oracle_lib.bf16_to_f64(w)
    for m in range(3):
        for v in range(5):
            assert got[m, v] == math.fsum(h[m, k] * ww[v, k] for k in range(8))


def test_orientation_closed_forms(oracle_lib):
    K, V = 16, 9
    _, w = wl.lm_head_inputs(1, K, V, seed=3)
    one = np.float32(1.0).view(np.uint32) >> np.uint32(16)
    hid = np.zeros((K, K), np.uint16)
    for k in range(K):
        hid[k, k] = one                                   # one-hot rows
    got = oracle_lib.lm_head(hid, w)
    np.testing.assert_array_equal(got, oracle_lib.bf16_to_f64(w).T)
    hid2, _ = wl.lm_head_inputs(4, K, 1, seed=4)
    ones = np.full((V, K), one, np.uint16)
    np.testing.assert_array_equal(oracle_lib.lm_head(hid2, ones),
                                  np.repeat(oracle_lib.bf16_to_f64(hid2).sum(1, keepdims=True), V, 1))


def test_rows_subset_and_widening(oracle_lib):
    hid, w = wl.lm_head_inputs(6, 24, 7, seed=5)
    full = oracle_lib.lm_head(hid, w)
    np.testing.assert_array_equal(oracle_lib.lm_head(hid, w, rows=[4, 1]), full[[4, 1]])
    x = np.float32([1.0, -2.5, 3.140625, 0.0])
    assert np.array_equal(oracle_lib.bf16_to_f64(wl.to_bf16_bits(x)), x.astype(np.float64))


def test_exact_inputs_give_fp32_exact_logits(oracle_lib):
    # The integer-valued inputs' logits are exact in fp32 in any summation
    # order: the fp64 logits round-trip through fp32, and fp32 sums taken
    # forwards, backwards and pairwise (numpy's blocked sum) all equal them.
    for K in (8, 136, 2688):
        hid, w = wl.lm_head_exact_inputs(5, K, 7, seed=K)
        ref = oracle_lib.lm_head(hid, w)
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)
        h = wl.bf16_bits_to_f32(hid)
        ww = wl.bf16_bits_to_f32(w)
        prod = h[:, None, :] * ww[None, :, :]           # exact products, fp32
        fwd = np.zeros(ref.shape, np.float32)
        bwd = np.zeros(ref.shape, np.float32)
        for k in range(K):
            fwd += prod[:, :, k]
            bwd += prod[:, :, K - 1 - k]
        np.testing.assert_array_equal(fwd, ref)
        np.testing.assert_array_equal(bwd, ref)
        np.testing.assert_array_equal(prod.sum(axis=2, dtype=np.float32), ref)
        # values on the stated grid, logits neither all zero nor overflowing
        assert set(np.unique(h * 8).astype(int)) <= set(range(-8, 9))
        assert 0.5 < ref.std() < 5.0
