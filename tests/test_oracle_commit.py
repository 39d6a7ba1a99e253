"""Pins of the CPU commit oracle against what the pages and mathematics fix.

"Nemotron-Labs-TwoTower" Section 2.2, Algorithm 2: each step predicts every
still-masked position, commits the confident ones and leaves the rest masked;
the block is complete within T steps. With a fixed budget of k commits per
block per step, T = ceil(L/k). Checks:

* the fp32 exponential behind the canonical key against libm exp (an ulp
  bound), and the quantiser against exact integer arithmetic;
* greedy prediction against numpy.argmax (first occurrence);
* the canonical key ordering against the float64 max-softmax probability
  wherever the float64 gap exceeds the quantisation bound;
* closed forms: equal logits give key V * 2^40; a lone dominant logit gives
  key 2^40 (confidence 1);
* a full denoising loop: exactly min(k, #masked) commits per block per step,
  no re-masking, untouched ids at uncommitted rows, fully unmasked after
  ceil(L/k) steps, one commit per step for k = 1 (mock autoregressive mode);
* with fixed logits the committed set after r steps is the first r*k rows of
  the (key, row) order; brute force over all k-subsets on a tiny block.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from block_diffusion_decoding_attn_b300 import workload as wl

TWO40 = 1 << 40
# measured maximum error of the own exponential over [-30, 0], in fp32 ulps
EXP_ULP_BOUND = 1.0


def _ulp32(x: float) -> float:
    return float(np.spacing(np.float32(x)))


def test_own_exp_against_libm(oracle_lib):
    xs = np.concatenate([
        -np.linspace(0, 30, 60001, dtype=np.float64),
        -np.geomspace(1e-9, 1, 5000),
        -np.array([np.float32(0.34657359), np.float32(0.34657360), np.float32(29.999998)]),
    ]).astype(np.float32)
    worst = 0.0
    for x in xs:
        e = oracle_lib.exp_own(float(x))
        ref = math.exp(float(x))
        worst = max(worst, abs(e - ref) / _ulp32(ref))
    assert worst <= EXP_ULP_BOUND, worst
    assert oracle_lib.exp_own(0.0) == 1.0
    assert oracle_lib.exp_own(-30.5) == 0.0


def _rhe(q: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even."""
    fl = math.floor(q)
    fr = q - fl
    return fl + (1 if fr > Fraction(1, 2) or (fr == Fraction(1, 2) and fl % 2) else 0)


def _rn32(q: Fraction) -> Fraction:
    """Round a nonzero rational in the fp32 normal range to fp32, ties to even (exact)."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    return s * _rhe(a / ulp) * ulp


def _quant_from_definition(x: float, n: int) -> int:
    """rint(2^40 * p(r) * 2^n) for a given n, every fp32 step done in exact
    rational arithmetic with one rounding per fused multiply-add."""
    ln2 = Fraction(0.69314718055994530942)   # the double nearest ln 2
    c1 = _rn32(ln2)
    c2 = _rn32(ln2 - c1)
    r = _rn32(-n * c1 + Fraction(x))
    r = _rn32(-n * c2 + r)
    c = [_rn32(1 / Fraction(math.factorial(j))) for j in range(8)]
    p = c[7]
    for j in range(6, -1, -1):
        p = _rn32(p * r + c[j])
    return _rhe(p * Fraction(2) ** (n + 40))


def test_reduction_n_is_one_rounding_of_the_exact_product(oracle_lib):
    # The reduction's n is the integer nearest the exact product x * RN32(1/ln 2),
    # rounded once (the Cody-Waite reduction as done with an FMA and a
    # 1.5 * 2^23 shifter, Muller, "Elementary Functions", Ch. 11). These x are
    # the fp32 values in [-30, 0] where rounding the product to fp32 first and
    # then to an integer gives another n: the product lies within half an fp32
    # ulp of a half-integer. The pin fixes the documented n, and the key term
    # that follows from it, against exact rational arithmetic.
    l2e = Fraction(float(np.float32(1.0 / 0.69314718055994530942)))
    cases = []
    for k in range(44):
        x0 = np.float32(-(k + 0.5) / float(l2e))
        for d in range(-40, 41):
            x = np.array([x0.view(np.int32) + d], np.int32).view(np.float32)[0]
            if not (-30.0 <= x <= 0.0):
                continue
            n_exact = _rhe(Fraction(float(x)) * l2e)
            n_twice = int(np.rint(np.float32(x) * np.float32(l2e)))  # RN32, then rint
            if n_exact != n_twice:
                cases.append((float(x), n_exact, n_twice))
    assert len(cases) >= 20
    assert any(x == float(np.float32(-1.0397208)) for x, _, _ in cases)
    differs = 0
    for x, n_exact, n_twice in cases:
        assert oracle_lib.exp_n(x) == n_exact, x
        q = oracle_lib.quant(x)
        assert q == _quant_from_definition(x, n_exact), x
        differs += q != _quant_from_definition(x, n_twice)
        # either way the term stays within the exponential's error bound
        assert abs(q - TWO40 * math.exp(x)) <= TWO40 * math.exp(x) * 2.0 ** -22 + 1
    assert differs >= 1  # the key terms themselves tell the two readings apart


def test_quantiser_is_exact_rounding_of_scaled_exp(oracle_lib):
    rng = np.random.default_rng(0)
    xs = np.concatenate([-rng.random(3000) * 30, -rng.random(500) * 1e-3, [0.0, -29.9, -30.0]])
    for x in xs.astype(np.float32):
        e = oracle_lib.exp_own(float(x))
        y = Fraction(e) * TWO40  # exact
        fl = math.floor(y)
        frac = y - fl
        expect = fl + (1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and fl % 2) else 0)
        assert oracle_lib.quant(float(x)) == expect
    assert oracle_lib.quant(0.0) == TWO40
    assert oracle_lib.quant(-31.0) == 0
    # monotone in x
    grid = np.linspace(-30, 0, 20001).astype(np.float32)
    q = [oracle_lib.quant(float(x)) for x in grid]
    assert all(a <= b for a, b in zip(q, q[1:]))


def test_prediction_is_first_argmax(oracle_lib):
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((40, 777)).astype(np.float32) * 2
    rows[3, [5, 600]] = 50.0            # tie -> lower index
    rows[4, :] = 0.0
    rows[4, 10] = -0.0                  # -0 == +0: first index wins
    rows[5, [0, 776]] = 99.0
    for r in rows:
        a, _ = oracle_lib.row_key(r)
        assert a == int(np.argmax(r))


def test_closed_forms(oracle_lib):
    V = 4096
    a, k = oracle_lib.row_key(np.full(V, 1.25, np.float32))
    assert (a, k) == (0, V * TWO40)      # confidence 1/V
    row = np.full(V, -100.0, np.float32)
    row[1234] = 7.0
    a, k = oracle_lib.row_key(row)
    assert (a, k) == (1234, TWO40)       # confidence exactly 1


def test_key_orders_like_float64_confidence(oracle_lib):
    w = wl.custom("conf", 4, 64, 1, 1, 8, 8, (0,) * 4, V=8192)
    lg = wl.logits(w, seed=5)
    lg[:8] = lg[8:16] * np.float32(1.0000001)  # near-ties
    keys = np.array([oracle_lib.row_key(r)[1] for r in lg], dtype=np.float64)
    l64 = lg.astype(np.float64)
    s64 = np.exp(l64 - l64.max(1, keepdims=True)).sum(1)  # 1 / max softmax prob
    # relative error of key/2^40 against the float64 sum
    bound = lg.shape[1] * 2.0 ** -41 + 4 * 2.0 ** -24
    rel = np.abs(keys / TWO40 - s64) / s64
    assert rel.max() <= bound, rel.max()
    order_ok = 0
    for i in range(len(lg)):
        for j in range(i + 1, len(lg)):
            gap = abs(s64[i] - s64[j]) / max(s64[i], s64[j])
            if gap > 2 * bound:
                assert (keys[i] < keys[j]) == (s64[i] < s64[j])
                order_ok += 1
    assert order_ok > 1000


def _loop_invariants(o, w, masked0, fresh=True, seed=0):
    tok = np.full(w.rows, -1, np.int32)
    masked = masked0.copy()
    steps = 0
    while masked.any():
        lg = wl.logits(w, seed=seed, step=steps if fresh else 0)
        t2, m2, keys, args = o.commit(lg, w.B, w.L, masked, w.k, tok)
        for b in range(w.B):
            sl = slice(b * w.L, (b + 1) * w.L)
            n = int(masked[sl].sum())
            assert int(masked[sl].sum() - m2[sl].sum()) == min(w.k, n)
        assert not np.any(m2 > masked)                       # never re-mask
        committed = (masked == 1) & (m2 == 0)
        np.testing.assert_array_equal(t2[~committed], tok[~committed])
        np.testing.assert_array_equal(t2[committed], args[committed])
        for r in np.nonzero(committed)[0]:
            assert t2[r] == int(np.argmax(lg[r]))
        tok, masked = t2, m2
        steps += 1
    return steps


@pytest.mark.parametrize("L,k", [(32, 4), (30, 4), (16, 1), (8, 8), (5, 9)])
def test_denoise_loop_invariants(oracle_lib, L, k):
    w = wl.custom(f"loop{L}_{k}", 3, L, 1, 1, 8, 8, (0,) * 3, V=512, k=k)
    steps = _loop_invariants(oracle_lib, w, np.ones(w.rows, np.uint8))
    assert steps == -(-L // k)


def test_ragged_mask_loop(oracle_lib):
    w = wl.custom("ragged", 4, 24, 1, 1, 8, 8, (0,) * 4, V=300, k=5)
    m0 = wl.random_mask(w, 0.6, seed=3)
    m0[:24] = 0  # one block fully committed already
    steps = _loop_invariants(oracle_lib, w, m0)
    assert steps == max(-(-int(m0[b * 24:(b + 1) * 24].sum()) // 5) for b in range(4))


def test_fixed_logits_closed_form(oracle_lib):
    w = wl.custom("fixed", 2, 20, 1, 1, 8, 8, (0, 0), V=640, k=3)
    lg = wl.logits(w, seed=9)
    lg[5] = lg[6]  # an exact tie: lower row first
    keys = [oracle_lib.row_key(r)[1] for r in lg]
    tok = np.full(w.rows, -1, np.int32)
    masked = np.ones(w.rows, np.uint8)
    for r in range(1, 8):
        tok, masked, _, _ = oracle_lib.commit(lg, w.B, w.L, masked, w.k, tok)
        for b in range(w.B):
            order = sorted(range(w.L), key=lambda i: (keys[b * w.L + i], i))
            want = set(order[:min(r * w.k, w.L)])
            got = {i for i in range(w.L) if masked[b * w.L + i] == 0}
            assert got == want
    assert keys[5] == keys[6]


def test_brute_force_subsets(oracle_lib):
    w = wl.custom("bf", 1, 7, 1, 1, 8, 8, (0,), V=64, k=3)
    lg = wl.logits(w, seed=4)
    lg[2] = lg[4]
    masked = np.array([1, 1, 1, 0, 1, 1, 1], np.uint8)
    tok, m2, _, _ = oracle_lib.commit(lg, 1, 7, masked, 3, np.full(7, -1, np.int32))
    keys = [oracle_lib.row_key(r)[1] for r in lg]
    cand = [i for i in range(7) if masked[i]]
    best = min(itertools.combinations(cand, 3),
               key=lambda s: sorted((keys[i], i) for i in s))
    assert {i for i in cand if m2[i] == 0} == set(best)
