/*
 * CPU oracle for the unmask/commit step -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code. It shares nothing with the CUDA path.
 *
 * Method followed: "Nemotron-Labs-TwoTower" Section 2.2, "Sampling", and
 * Algorithm 2 (single-block confidence unmasking): at each step the denoiser
 * predicts every still-masked position in parallel, the confident predictions
 * are committed, and the rest stay masked. ConfidenceSample is not spelled out
 * on the page; the reading used here (a fixed budget of k commits per block per
 * step) is Algorithm 2 with a threshold above 1 and T = L/k steps.
 *
 * Per still-masked row r (a scalar loop, in the order below):
 *   1. m = max_v l[r][v]; a = lowest v with l[r][v] == m (greedy prediction).
 *   2. confidence = max softmax probability = 1 / sum_v exp(l[r][v] - m),
 *      computed as the canonical fixed-point key
 *          key = sum_v q(RN32(l[r][v] - m)),   q(x) = rint(2^40 * e(x))
 *      with e the fp32 exponential defined in own_exp below; the integer sum
 *      does not depend on summation order. Smaller key = more confident.
 *   3. Per block: sort the masked rows by (key ascending, row ascending) and
 *      commit the first min(k, #masked): tok[r] = a, masked[r] = 0.
 *
 * The exponential (a reading: the page only says "confidence"):
 *   x < -30          -> q = 0  (2^40 * exp(-30) < 0.11 rounds to 0 anyway)
 *   n = x * LOG2E rounded to the nearest integer, ties to even, from the exact
 *       product: nb = fma(x, LOG2E, 1.5 * 2^23) (one rounding), n = nb - 1.5 * 2^23
 *   r = fma(-n, C1, x); r = fma(-n, C2, r)      (Cody and Waite reduction)
 *   p = c7; p = fma(p, r, c_j) for j = 6..0     (Taylor series, c_j = 1/j!)
 *   q = round-half-even(p * 2^(n+40))           (exact power-of-two scale)
 * with LOG2E = RN32(1/ln 2), C1 = RN32(ln 2), C2 = RN32(ln 2 - C1),
 * c_j = RN32(1/j!). fmaf is the correctly rounded fused multiply-add.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LN2_D 0.69314718055994530942
static const float LOG2E_F = (float)(1.0 / LN2_D);
static const float C1_F = (float)LN2_D;

static float c2_f(void) { return (float)(LN2_D - (double)C1_F); }

/* n = nearest integer (ties to even) to the exact product x * LOG2E; |n| < 2^22.
 * This is the Cody-Waite choice of n: the integer nearest to x / ln 2 as
 * approximated by x * RN32(1/ln 2), rounded once. Rounding the product to fp32
 * first and then to an integer would round twice; the two differ for x whose
 * product lies within half an fp32 ulp of a half-integer (e.g. x = -1.0397208,
 * where RN32(x * LOG2E) = -1.5 exactly and the exact product is above it). */
static float reduce_n(float x) {
    const float magic = 12582912.0f; /* 1.5 * 2^23: sums in [2^23, 2^24) have ulp 1 */
    const float nb = fmaf(x, LOG2E_F, magic);
    return nb - magic;
}

/* The n of the reduction step for x (exposed so that the tests can pin which
 * rounding defines it). */
float tt_oracle_exp_n(float x) { return reduce_n(x); }

/* e(x) for -30 <= x <= 0 as a float: p(r) * 2^n. Returns 0 below -30. */
float tt_oracle_exp_own(float x) {
    if (x < -30.0f) return 0.0f;
    const float n = reduce_n(x);
    float r = fmaf(-n, C1_F, x);
    r = fmaf(-n, c2_f(), r);
    static const double inv_fact[8] = {1.0, 1.0, 1.0 / 2, 1.0 / 6, 1.0 / 24, 1.0 / 120, 1.0 / 720,
                                       1.0 / 5040};
    float p = (float)inv_fact[7];
    for (int j = 6; j >= 0; --j) p = fmaf(p, r, (float)inv_fact[j]);
    return ldexpf(p, (int)n);
}

/* q(x) = rint(2^40 * e(x)). */
uint64_t tt_oracle_quant(float x) {
    if (x < -30.0f) return 0;
    const float n = reduce_n(x);
    float r = fmaf(-n, C1_F, x);
    r = fmaf(-n, c2_f(), r);
    static const double inv_fact[8] = {1.0, 1.0, 1.0 / 2, 1.0 / 6, 1.0 / 24, 1.0 / 120, 1.0 / 720,
                                       1.0 / 5040};
    float p = (float)inv_fact[7];
    for (int j = 6; j >= 0; --j) p = fmaf(p, r, (float)inv_fact[j]);
    const float y = ldexpf(p, (int)n + 40); /* exact: a power-of-two scale of a normal */
    return (uint64_t)rintf(y);
}

/* Greedy prediction and canonical confidence key of one row. */
void tt_oracle_row_key(const float* row, long V, int32_t* arg, uint64_t* key) {
    float m = row[0];
    long a = 0;
    for (long v = 1; v < V; ++v)
        if (row[v] > m) { m = row[v]; a = v; } /* strict: first occurrence wins */
    uint64_t s = 0;
    for (long v = 0; v < V; ++v) {
        const float x = row[v] - m; /* one fp32 subtraction, round to nearest */
        s += tt_oracle_quant(x);
    }
    *arg = (int32_t)a;
    *key = s;
}

typedef struct { uint64_t key; int32_t row; } keyed_row;

static int cmp_keyed(const void* pa, const void* pb) {
    const keyed_row* a = (const keyed_row*)pa;
    const keyed_row* b = (const keyed_row*)pb;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    return (a->row > b->row) - (a->row < b->row);
}

/*
 * One commit step over B blocks of L rows. tok is updated in place at the
 * committed rows only; masked_out receives the new mask (may equal masked).
 * keys_out / args_out (may be NULL) receive the key and prediction of every
 * masked row (untouched for unmasked rows). Returns 0, or -1 on bad arguments.
 */
int tt_oracle_commit(const float* logits, int B, int L, long V, const uint8_t* masked, int k,
                     int32_t* tok, uint8_t* masked_out, uint64_t* keys_out,
                     int32_t* args_out, int nthreads) {
    if (B < 0 || L < 0 || V < 1 || k < 1) return -1;
    const long R = (long)B * L;
    uint64_t* key = (uint64_t*)malloc(sizeof(uint64_t) * (R ? R : 1));
    int32_t* arg = (int32_t*)malloc(sizeof(int32_t) * (R ? R : 1));
    uint8_t* m_in = (uint8_t*)malloc(R ? R : 1);
    keyed_row* buf = (keyed_row*)malloc(sizeof(keyed_row) * (L ? L : 1));
    if (!key || !arg || !m_in || !buf) { free(key); free(arg); free(m_in); free(buf); return -1; }
    memcpy(m_in, masked, R);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < R; ++r)
        if (m_in[r]) tt_oracle_row_key(logits + (size_t)r * V, V, &arg[r], &key[r]);

    for (int b = 0; b < B; ++b) {
        int n = 0;
        for (int i = 0; i < L; ++i) {
            const long r = (long)b * L + i;
            if (m_in[r]) { buf[n].key = key[r]; buf[n].row = i; ++n; }
        }
        qsort(buf, n, sizeof(keyed_row), cmp_keyed);
        for (int i = 0; i < L; ++i) masked_out[(long)b * L + i] = m_in[(long)b * L + i];
        const int c = n < k ? n : k;
        for (int j = 0; j < c; ++j) {
            const long r = (long)b * L + buf[j].row;
            tok[r] = arg[r];
            masked_out[r] = 0;
        }
    }
    for (long r = 0; r < R; ++r)
        if (m_in[r]) {
            if (keys_out) keys_out[r] = key[r];
            if (args_out) args_out[r] = arg[r];
        }
    free(key); free(arg); free(m_in); free(buf);
    return 0;
}

/*
 * Confidence above a threshold (Section 2.2, Algorithm 2: a prediction whose
 * confidence exceeds gamma is committed): confidence = 2^40 / key, so conf > gamma is
 * gamma * key < 2^40, decided in exact arithmetic. gamma = f * 2^e with f in
 * [0.5, 1), and m = f * 2^53 is an integer, so the test is
 * m * key < 2^(93 - e) on 128-bit integers.
 */
int tt_oracle_conf_above(uint64_t key, double gamma) {
    if (!(gamma > 0.0)) return 1;   /* every confidence is positive */
    if (isinf(gamma)) return 0;
    int e;
    const double f = frexp(gamma, &e);
    const unsigned __int128 m = (unsigned __int128)(uint64_t)ldexp(f, 53);
    const int sh = 93 - e;
    if (sh >= 127) return 1;        /* m * key < 2^110 <= 2^sh */
    if (sh <= 0) return 0;
    return m * (unsigned __int128)key < ((unsigned __int128)1 << sh);
}

/*
 * One step of threshold unmasking: per block, commit every masked row whose
 * confidence exceeds gamma, and at least ceil(n / steps_left) of the n masked
 * rows (the most confident first), so that a block is complete after
 * steps_left more steps. Rows are ranked by (key ascending, row ascending).
 * Same arguments and results as tt_oracle_commit otherwise.
 */
int tt_oracle_commit_threshold(const float* logits, int B, int L, long V, const uint8_t* masked,
                               double gamma, int steps_left, int32_t* tok, uint8_t* masked_out,
                               uint64_t* keys_out, int32_t* args_out, int nthreads) {
    if (B < 0 || L < 0 || V < 1 || steps_left < 1 || isnan(gamma)) return -1;
    const long R = (long)B * L;
    uint64_t* key = (uint64_t*)malloc(sizeof(uint64_t) * (R ? R : 1));
    int32_t* arg = (int32_t*)malloc(sizeof(int32_t) * (R ? R : 1));
    uint8_t* m_in = (uint8_t*)malloc(R ? R : 1);
    keyed_row* buf = (keyed_row*)malloc(sizeof(keyed_row) * (L ? L : 1));
    if (!key || !arg || !m_in || !buf) { free(key); free(arg); free(m_in); free(buf); return -1; }
    memcpy(m_in, masked, R);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < R; ++r)
        if (m_in[r]) tt_oracle_row_key(logits + (size_t)r * V, V, &arg[r], &key[r]);

    for (int b = 0; b < B; ++b) {
        int n = 0, above = 0;
        for (int i = 0; i < L; ++i) {
            const long r = (long)b * L + i;
            if (m_in[r]) {
                buf[n].key = key[r];
                buf[n].row = i;
                ++n;
                above += tt_oracle_conf_above(key[r], gamma);
            }
        }
        qsort(buf, n, sizeof(keyed_row), cmp_keyed);
        for (int i = 0; i < L; ++i) masked_out[(long)b * L + i] = m_in[(long)b * L + i];
        const int floor_k = (n + steps_left - 1) / steps_left;
        const int c = above > floor_k ? above : floor_k;
        for (int j = 0; j < c && j < n; ++j) {
            const long r = (long)b * L + buf[j].row;
            tok[r] = arg[r];
            masked_out[r] = 0;
        }
    }
    for (long r = 0; r < R; ++r)
        if (m_in[r]) {
            if (keys_out) keys_out[r] = key[r];
            if (args_out) args_out[r] = arg[r];
        }
    free(key); free(arg); free(m_in); free(buf);
    return 0;
}
