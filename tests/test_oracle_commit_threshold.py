"""Pins of the CPU oracle's threshold unmasking against what the pages and
exact arithmetic fix.

"Nemotron-Labs-TwoTower" Section 2.2, Algorithm 2: at each step the masked
predictions whose confidence is above gamma are committed and the uncertain
ones stay masked, and the block must be complete within T steps (read here as
a floor of ceil(#masked / steps_left) commits per step, steps_left = T - r + 1).
Checks:

* the "confidence > gamma" test (confidence = 2^40 / key) against exact
  rational arithmetic (Python fractions), including gammas that hit a key's
  confidence exactly;
* per block and step: every masked row above gamma commits, at least
  ceil(n / steps_left) rows commit, the committed rows are the most confident
  ones (a prefix of the (key, row) order), nothing is re-masked;
* a full denoising loop with steps_left = T - r + 1 ends fully unmasked after
  exactly T steps, whatever gamma;
* special cases: gamma <= 0 commits every masked row; gamma > 1 (no
  confidence exceeds it) commits exactly the floor, which equals the fixed
  budget k when steps_left = ceil(n / k).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

TWO40 = 1 << 40


def _exact_above(key: int, gamma: float) -> bool:
    if gamma <= 0:
        return True
    if math.isinf(gamma):
        return False
    return Fraction(gamma) * key < TWO40


def test_conf_above_is_exact(oracle_lib):
    rng = np.random.default_rng(5)
    keys = [TWO40, TWO40 + 1, 2 * TWO40 - 1, 2 * TWO40, 3 * TWO40 + 7, (1 << 57) - 1]
    keys += [int(k) for k in rng.integers(TWO40, 1 << 57, 400, dtype=np.uint64)]
    gammas = [0.0, -0.5, 1.0, 0.5, 1.0 / 3.0, 0.999999, 2.0, math.inf, 1e-300, 1e-17, 0.8]
    gammas += list(rng.random(60))
    for key in keys:
        # gammas right at, just below and just above this key's confidence
        c = TWO40 / key
        for g in gammas + [c, math.nextafter(c, 0.0), math.nextafter(c, 2.0)]:
            assert oracle_lib.conf_above(key, g) == _exact_above(key, g), (key, g)


def _block_checks(oracle_lib, lg, B, L, masked, gamma, steps_left, tok):
    to, mo, keys, args = oracle_lib.commit_threshold(lg, B, L, masked, gamma, steps_left, tok)
    for b in range(B):
        sl = slice(b * L, (b + 1) * L)
        m_in, m_out = masked[sl], mo[sl]
        rows = [i for i in range(L) if m_in[i]]
        n = len(rows)
        committed = [i for i in rows if m_out[i] == 0]
        assert all(m_out[i] == 0 for i in range(L) if not m_in[i])  # never re-masked
        order = sorted(rows, key=lambda i: (int(keys[b * L + i]), i))
        above = [i for i in rows if _exact_above(int(keys[b * L + i]), gamma)]
        want = max(len(above), -(-n // steps_left)) if n else 0
        assert sorted(committed) == sorted(order[:want])       # most confident first
        assert set(above) <= set(committed)                    # everything above gamma
        for i in committed:                                    # ids = greedy predictions
            assert to[b * L + i] == args[b * L + i] == int(np.argmax(lg[b * L + i]))
        for i in range(L):                                     # others untouched
            if i not in committed:
                assert to[b * L + i] == tok[b * L + i]
    return to, mo, keys


@pytest.mark.parametrize("gamma", [0.0, 0.02, 0.05, 0.3, 0.8, 1.5])
@pytest.mark.parametrize("steps_left", [1, 2, 3, 8])
def test_single_step_rule(oracle_lib, gamma, steps_left):
    w = wl.custom("thr", 3, 24, 1, 1, 8, 8, (0, 0, 0), V=256, k=4, logit_std=3.0)
    lg = wl.logits(w, seed=21)
    masked = wl.random_mask(w, 0.7, seed=4)
    tok = np.arange(w.rows, dtype=np.int32) - 50
    _block_checks(oracle_lib, lg, w.B, w.L, masked, gamma, steps_left, tok)


@pytest.mark.parametrize("gamma", [0.9, 0.1, 0.03])
def test_denoise_loop_completes_in_T_steps(oracle_lib, gamma):
    w = wl.custom("thr_loop", 2, 32, 1, 1, 8, 8, (0, 0), V=512, k=4, logit_std=3.0)
    T = 6
    tok = np.full(w.rows, -1, np.int32)
    masked = np.ones(w.rows, np.uint8)
    for r in range(1, T + 1):
        lg = wl.logits(w, seed=3, step=r)
        tok, masked, _ = _block_checks(oracle_lib, lg, w.B, w.L, masked, gamma, T - r + 1, tok)
        if r < T:
            # the floor alone leaves exactly L - r * ceil-share masked at worst
            assert masked.sum() <= w.rows
    assert not masked.any()


def test_special_cases(oracle_lib):
    w = wl.custom("thr_sp", 2, 40, 1, 1, 8, 8, (0, 0), V=1024, k=5)
    lg = wl.logits(w, seed=8)
    masked = np.ones(w.rows, np.uint8)
    tok = np.full(w.rows, -1, np.int32)
    _, mo, _, _ = oracle_lib.commit_threshold(lg, w.B, w.L, masked, 0.0, 7, tok)
    assert not mo.any()                                        # gamma <= 0: all commit
    # gamma above 1: the floor alone; with steps_left = L / k it is the fixed budget k
    t1, m1, _, _ = oracle_lib.commit_threshold(lg, w.B, w.L, masked, 1.5, w.L // w.k, tok)
    t2, m2, _, _ = oracle_lib.commit(lg, w.B, w.L, masked, w.k, tok)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(m1, m2)
