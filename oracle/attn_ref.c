/*
 * CPU oracle for the denoiser's block attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this code. It shares nothing with the CUDA path.
 *
 * Definition followed: "Nemotron-Labs-TwoTower" Section 2.1, "Bidirectional
 * Attention", Eq. (1):
 *
 *   Attn(Q_b^(i), [K_<b^ctx,(i); K_b^den,(i)], [V_<b^ctx,(i); V_b^den,(i)])
 *
 * Each query of the noisy block takes one softmax over the concatenation of
 * the context tower's layer-i keys for all clean positions before the block
 * and the denoiser's own keys for the block, with no mask inside the block.
 * Causality towards past clean blocks holds because the cache only holds past
 * positions.
 *
 * Causal variant (tt_oracle_block_attn_causal): the context tower's pass
 * over a committed block (Section 2.1, Algorithm 1: once a block is committed,
 * the context tower runs its tokens causally to update its caches). Block query l
 * takes its softmax over the cache positions and block keys 0..l only, i.e.
 * the key list above cut after block key l.
 *
 * Readings (the pages are silent on these): query head h uses KV head
 * floor(h / (Hq/Hkv)); the score scale is a parameter (1/sqrt(D) by default);
 * no positional encoding is applied here.
 *
 * Arithmetic: bf16 inputs widened exactly to double; every sum in double;
 * plain loops in the order of the definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline double bf16_to_double(uint16_t b) {
    union { uint32_t u; float f; } v;
    v.u = ((uint32_t)b) << 16;
    return (double)v.f;
}

/* One output row: batch b, block position l, query head h. */
static void attn_row(int L, int Hq, int Hkv, int D, int ctx_cap, double scale,
                     const uint16_t* q, const uint16_t* k_blk, const uint16_t* v_blk,
                     const uint16_t* k_ctx, const uint16_t* v_ctx, int C, int b, int l,
                     int h, int causal, double* s, double* out) {
    const int G = Hq / Hkv;
    const int kv = h / G;
    /* concatenated key list: context, then block (causal: block keys 0..l) */
    const int N = C + (causal ? l + 1 : L);
    const uint16_t* qr = q + (((size_t)b * L + l) * Hq + h) * D;

    /* scores s_j = scale * <q, k_j> */
    for (int j = 0; j < N; ++j) {
        const uint16_t* kr = (j < C)
            ? k_ctx + (((size_t)b * Hkv + kv) * ctx_cap + j) * D
            : k_blk + (((size_t)b * L + (j - C)) * Hkv + kv) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
        s[j] = scale * acc;
    }
    /* softmax over the whole list */
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) if (s[j] > mx) mx = s[j];
    double den = 0.0;
    for (int j = 0; j < N; ++j) { s[j] = exp(s[j] - mx); den += s[j]; }
    /* out = sum_j p_j v_j */
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = 0; j < N; ++j) {
        const uint16_t* vr = (j < C)
            ? v_ctx + (((size_t)b * Hkv + kv) * ctx_cap + j) * D
            : v_blk + (((size_t)b * L + (j - C)) * Hkv + kv) * D;
        const double p = s[j] / den;
        for (int d = 0; d < D; ++d) out[d] += p * bf16_to_double(vr[d]);
    }
}

/*
 * rows == NULL: every (b, l, h) row, out is [B][L][Hq][D].
 * rows != NULL: nrows triples (b, l, h), out is [nrows][D].
 * Returns 0, or -1 on an argument error (ctx_len outside [0, ctx_cap],
 * Hq not a multiple of Hkv, a row triple out of range).
 */
static int block_attn_rows(int B, int L, int Hq, int Hkv, int D, int ctx_cap, double scale,
                           const uint16_t* q, const uint16_t* k_blk, const uint16_t* v_blk,
                           const uint16_t* k_ctx, const uint16_t* v_ctx,
                           const int32_t* ctx_len, int nrows, const int32_t* rows,
                           double* out, int nthreads, int causal) {
    if (B < 0 || L < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv) return -1;
    for (int b = 0; b < B; ++b)
        if (ctx_len[b] < 0 || ctx_len[b] > ctx_cap) return -1;
    const long total = rows ? nrows : (long)B * L * Hq;
    if (rows)
        for (long i = 0; i < total; ++i) {
            const int b = rows[3 * i], l = rows[3 * i + 1], h = rows[3 * i + 2];
            if (b < 0 || b >= B || l < 0 || l >= L || h < 0 || h >= Hq) return -1;
        }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * ((size_t)ctx_cap + L));
        if (!s) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long i = 0; i < total; ++i) {
                int b, l, h;
                if (rows) { b = rows[3 * i]; l = rows[3 * i + 1]; h = rows[3 * i + 2]; }
                else { b = (int)(i / ((long)L * Hq)); l = (int)((i / Hq) % L); h = (int)(i % Hq); }
                attn_row(L, Hq, Hkv, D, ctx_cap, scale, q, k_blk, v_blk, k_ctx, v_ctx,
                         ctx_len[b], b, l, h, causal, s, out + (size_t)i * D);
            }
            free(s);
        }
    }
    return err ? -1 : 0;
}

int tt_oracle_block_attn(int B, int L, int Hq, int Hkv, int D, int ctx_cap, double scale,
                         const uint16_t* q, const uint16_t* k_blk, const uint16_t* v_blk,
                         const uint16_t* k_ctx, const uint16_t* v_ctx,
                         const int32_t* ctx_len, int nrows, const int32_t* rows,
                         double* out, int nthreads) {
    return block_attn_rows(B, L, Hq, Hkv, D, ctx_cap, scale, q, k_blk, v_blk, k_ctx, v_ctx,
                           ctx_len, nrows, rows, out, nthreads, 0);
}

int tt_oracle_block_attn_causal(int B, int L, int Hq, int Hkv, int D, int ctx_cap, double scale,
                                const uint16_t* q, const uint16_t* k_blk, const uint16_t* v_blk,
                                const uint16_t* k_ctx, const uint16_t* v_ctx,
                                const int32_t* ctx_len, int nrows, const int32_t* rows,
                                double* out, int nthreads) {
    return block_attn_rows(B, L, Hq, Hkv, D, ctx_cap, scale, q, k_blk, v_blk, k_ctx, v_ctx,
                           ctx_len, nrows, rows, out, nthreads, 1);
}
