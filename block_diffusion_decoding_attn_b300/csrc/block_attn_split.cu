// Block attention of the TwoTower denoiser ("Nemotron-Labs-TwoTower",
// Section 2.1, Eq. 1), one-unit-per-CTA schedule: the same computation as
// block_attn.cu (including its causal variant and training layout), with the
// work cut on the host instead of in the kernel. It is the faster schedule
// when units are short or of equal length (the library picks it by shape;
// see tt_api.cu).
//
// One CTA owns one work unit: (sequence b, KV head, pair of 128-row query
// tiles, KV split). The host picks the split count from the cache capacity
// (minimising waves times tiles per split, one CTA per SM); a split past the
// end of its sequence's keys exits at once. Sequences whose keys fit one
// split write their output directly; the others write fp32 partials
// (running max, running sum, O) that attn_merge_kernel combines, launched as
// a programmatic dependent of this grid.
//
// Warp roles (320 threads), TMEM columns and the ping-pong of the two query
// tiles on the tensor core are those of block_attn.cu: warps 0-7 softmax
// (one query row per thread), warp 8 TMA producer (Q once, then K_j, V_j into
// a 5-slot ring), warp 9 MMA issuer and TMEM owner.
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

constexpr int kRing = 5;               // K/V tile slots (K_j and V_j alternate)
constexpr float kRescaleThresh = 8.0f; // log2 units

template <int D>
struct SplitLayout {
    static constexpr int kTileBytes = kTile * D * 2;  // a Q, K or V tile (bf16)
    static constexpr int kAtomBytes = kTile * 128;    // one 64-column swizzle atom column
    static constexpr int kQ = 0;                      // Q_A, then Q_B
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBar = kRingOff + kRing * kTileBytes;
    // q_full, full[kRing], empty[kRing], s_full[2], p_full[2], o_final[2], drain
    static constexpr int kNumBars = 1 + 2 * kRing + 7;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack for the 1024-byte alignment
};

struct KvTile {
    int is_ctx;  // 1: context-cache tile, 0: block tile
    int base;    // first key (cache position or block position)
    int valid;   // keys of this tile that exist (1..128)
};

__device__ __forceinline__ KvTile kv_tile(int j, int nc, int C, int L) {
    if (j < nc) return {1, j * kTile, min(kTile, C - j * kTile)};
    const int jb = j - nc;
    return {0, jb * kTile, min(kTile, L - jb * kTile)};
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    block_attn_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kc,
                      const __grid_constant__ CUtensorMap tm_vc,
                      const __grid_constant__ CUtensorMap tm_kb,
                      const __grid_constant__ CUtensorMap tm_vb, const AttnSplitParams p) {
    using Lay = SplitLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x % p.n_pairs;
    const int split = blockIdx.x / p.n_pairs;
    const int kvh = blockIdx.y;
    int b = blockIdx.z;
    if (p.ctx_group) {
        // Training layout: block j of a sequence sees j * L cache keys, so the
        // grid takes block j of every sequence for j descending (longest
        // first), which keeps the last wave short.
        const int nseq = static_cast<int>(gridDim.z) / p.ctx_group;
        const int j = p.ctx_group - 1 - static_cast<int>(blockIdx.z) / nseq;
        b = static_cast<int>(blockIdx.z) % nseq * p.ctx_group + j;
    }

    int C = p.ctx_group ? (b % p.ctx_group) * p.L : p.ctx_len[b];
    if (C < 0 || C > p.ctx_cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) atomicOr(p.status, kDevCtxLenRange);
        C = C < 0 ? 0 : p.ctx_cap;
    }
    const int cache_b = p.ctx_group ? b / p.ctx_group : b;  // which cache sequence b reads
    const int nc = (C + kTile - 1) / kTile;
    const int nt = nc + p.nblk;
    const int t0 = split * p.chunk;
    if (t0 >= nt) return;  // this split is past the end of sequence b's keys
    const int n = min(nt, t0 + p.chunk) - t0;
    const int nsplit_b = (nt + p.chunk - 1) / p.chunk;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::kBar);
    uint64_t* q_full = bars;
    uint64_t* full = bars + 1;
    uint64_t* empty = full + kRing;
    uint64_t* s_full = empty + kRing;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_final = p_full + 2;
    uint64_t* drain = o_final + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 128);
            mbar_init(&o_final[s], 1);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t limit = p.timeout_ns;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_kc);
            tma_prefetch_desc(&tm_vc);
            tma_prefetch_desc(&tm_kb);
            tma_prefetch_desc(&tm_vb);
            mbar_arrive_expect_tx(q_full, 2 * Lay::kTileBytes);
            const int rows_l = kTile / p.G;  // block positions per query tile
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_5d(sm + Lay::kQ + t * Lay::kTileBytes + c * Lay::kAtomBytes, &tm_q,
                                q_full, c * 64, 0, kvh, (2 * pair + t) * rows_l, b);
            bool ok = true;
            int issued = 0;  // ring loads issued: K_j is load 2j, V_j is load 2j+1
            for (int li = 0; li < 2 * n; ++li) {
                const int slot = li % kRing;
                if (li >= kRing && !mbar_wait(&empty[slot], ((li / kRing) & 1) ^ 1, limit)) {
                    ok = false;
                    break;
                }
                const KvTile t = kv_tile(t0 + (li >> 1), nc, C, p.L);
                const bool is_v = li & 1;
                uint8_t* dst = sm + Lay::kRingOff + slot * Lay::kTileBytes;
                mbar_arrive_expect_tx(&full[slot], Lay::kTileBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if (t.is_ctx)
                        tma_load_3d(dst + c * Lay::kAtomBytes, is_v ? &tm_vc : &tm_kc, &full[slot],
                                    c * 64, t.base, cache_b * p.Hkv + kvh);
                    else
                        tma_load_4d(dst + c * Lay::kAtomBytes, is_v ? &tm_vb : &tm_kb, &full[slot],
                                    c * 64, kvh, t.base, b);
                }
                issued = li + 1;
            }
            if (!ok) atomicOr(p.status, kDevWaitTimeout);
            // Let the copies already issued land before the CTA can exit (a load
            // is issued only once the load kRing before it was consumed, so at
            // most the last kRing can be in flight; after a normal run they
            // have all landed). Also after a timeout of another role.
            const uint64_t dl = drain_limit(limit);
            mbar_wait(q_full, 0, dl);
            for (int li = issued - kRing < 0 ? 0 : issued - kRing; li < issued; ++li)
                mbar_wait(&full[li % kRing], (li / kRing) & 1, dl);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16(kTile, kTile, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, 0, 1);
        const uint32_t sq = smem_u32(sm + Lay::kQ);
        const uint32_t ring = smem_u32(sm + Lay::kRingOff);
        const uint32_t col_s[2] = {0u, 2u * kTile};
        const uint32_t col_o[2] = {static_cast<uint32_t>(kTile), 3u * kTile};
        auto wait_slot = [&](int li) {
            return mbar_wait(&full[li % kRing], (li / kRing) & 1, limit);
        };
        // S_X = Q_X K^T for the K tile in ring load li
        auto issue_s = [&](int x, int li) {
            const uint32_t sk = ring + (li % kRing) * Lay::kTileBytes;
            const uint32_t sqx = sq + x * Lay::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * Lay::kAtomBytes + (kk & 3) * 32;
                tc_mma_ss(tmem + col_s[x], sdesc_sw128(sqx + off, 16, 1024),
                          sdesc_sw128(sk + off, 16, 1024), idesc_qk, kk > 0);
            }
        };
        // O_X (+)= P_X V for the V tile in ring load li
        auto issue_pv = [&](int x, int li, bool first) {
            const uint32_t sv = ring + (li % kRing) * Lay::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
                // V is MN-major (d contiguous): 16 keys = two 8-row atoms; the
                // next 64 columns of d sit one atom column further.
                const uint64_t bd = sdesc_sw128(sv + kk * 2048, Lay::kAtomBytes, 1024);
                tc_mma_ts(tmem + col_o[x], tmem + col_s[x] + kk * 8, bd, idesc_pv,
                          (!first || kk > 0) ? 1u : 0u);
            }
        };
        auto zero_tail = [&](int j, int li) {
            // Cache rows past ctx_len may hold anything (even NaN); P is 0
            // there, but 0 * NaN is not, so zero those V rows.
            const KvTile kt = kv_tile(t0 + j, nc, C, p.L);
            if (kt.is_ctx && kt.valid < kTile) {
                uint8_t* sv = sm + Lay::kRingOff + (li % kRing) * Lay::kTileBytes;
                const int rows = kTile - kt.valid;
                for (int u = lane; u < rows * 8 * (D / 64); u += 32) {
                    const int c = u / (rows * 8);
                    const int rem = u % (rows * 8);
                    const int r = kt.valid + rem / 8;
                    *reinterpret_cast<uint4*>(sv + c * Lay::kAtomBytes + r * 128 + (rem % 8) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
        };

        bool ok = mbar_wait(q_full, 0, limit) && wait_slot(0);
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
                issue_s(0, 0);
                tc_commit(&s_full[0]);
                issue_s(1, 0);
                tc_commit(&s_full[1]);
                tc_commit(&empty[0]);
            }
            __syncwarp();
        }
        for (int j = 0; j < n && ok; ++j) {
            const int lv = 2 * j + 1, lk = 2 * j + 2;
            const bool more = j + 1 < n;
            // ---- tile A: every input of its group (P_A, V_j, K_j+1) is in
            // before the first of its MMAs, so that P V and the next QK^T go to
            // the tensor core back to back
            if (!mbar_wait(&p_full[0], j & 1, limit) || !wait_slot(lv) || (more && !wait_slot(lk))) {
                ok = false;
                break;
            }
            zero_tail(j, lv);
            tc_fence_after();
            if (lane == 0) {
                issue_pv(0, lv, j == 0);
                if (more) {
                    issue_s(0, lk);
                    tc_commit(&s_full[0]);
                } else {
                    tc_commit(&o_final[0]);
                }
            }
            __syncwarp();
            // ---- tile B
            if (!mbar_wait(&p_full[1], j & 1, limit)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) {
                issue_pv(1, lv, j == 0);
                tc_commit(&empty[lv % kRing]);
                if (more) {
                    issue_s(1, lk);
                    tc_commit(&s_full[1]);
                    tc_commit(&empty[lk % kRing]);
                } else {
                    tc_commit(&o_final[1]);
                }
            }
            __syncwarp();
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        // No MMA may still be running when the TMEM is released.
        if (lane == 0) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, drain_limit(limit));
    } else {
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;               // query tile
        const int row = (warp & 3) * 32 + lane;  // TMEM lane = row of the tile
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t ts = tmem + lane_off + (x ? 2u * kTile : 0u);
        const uint32_t to = tmem + lane_off + (x ? 3u * kTile : static_cast<uint32_t>(kTile));
        const float sl2 = p.scale_log2;
        // block position of this thread's query row (rows past G*L are padding)
        const int lq = ((2 * pair + x) * kTile + row) / p.G;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], j & 1, limit));
            if (!ok) break;
            tc_fence_after();
            float s[kTile];
            {
                uint32_t r[kTile];
                tmem_ld128(ts, r);
#pragma unroll
                for (int c = 0; c < kTile; ++c) s[c] = __uint_as_float(r[c]);
            }
            const KvTile kt = kv_tile(t0 + j, nc, C, p.L);
            // keys of this tile the row sees: the tile's keys, and in the causal
            // variant only block keys up to the row's own position (maybe none)
            const int lim = (p.causal && !kt.is_ctx) ? min(kt.valid, lq + 1 - kt.base) : kt.valid;
            if (lim < kTile) {
#pragma unroll
                for (int c = 0; c < kTile; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
            }
            const float mx = row_max128(s);
            const float m_tile = mx * sl2;
            if (j == 0) {
                m_run = m_tile;
            } else if (__any_sync(0xffffffffu, m_tile > m_run + kRescaleThresh)) {
                // Warp-uniform (the TMEM accesses are warp-collective): every
                // lane moves to its new max; alpha is 1 where nothing changed.
                // O_X is final for KV tile j-1 (S_X(j) completed after it).
                const float m_new = fmaxf(m_run, m_tile);
                const float alpha = ex2_approx(m_run - m_new);
                m_run = m_new;
                l_run *= alpha;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t r[32];
                    tmem_ld32(to + c4 * 32, r);
#pragma unroll
                    for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                    tmem_st32(to + c4 * 32, r);
                }
            }
            // A row that has seen no key yet (causal variant) has m_run = -inf:
            // its P is exp2(-inf) = 0 rather than exp2(-inf + inf).
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};  // 8 sum chains
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // P in two halves of 64 keys (32 columns each)
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    float a0, a1;
                    fma2(a0, a1, s[h * 64 + c], s[h * 64 + c + 1], sl2, sl2, neg_m, neg_m);
                    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                    const int q = (c >> 1) & 3;
                    add2(sa[q], sb[q], sa[q], sb[q], e0, e1);
                    pk[c >> 1] = pack_bf16x2(e0, e1);
                }
                tmem_st32(ts + h * 32, pk);  // P over the first 64 columns of S_X
            }
            l_run += ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
            tc_fence_before();
            mbar_arrive(&p_full[x]);
        }
        // The split merge (launched as a programmatic dependent) may start
        // launching now; it still waits for this grid's completion.
        if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_final[x], 0, limit));
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kDevWaitTimeout);
        } else {
            tc_fence_after();
            const int m = (2 * pair + x) * kTile + row;
            const int l = m / p.G, g = m % p.G;
            const bool live = l < p.L;
            uint32_t r[kTile];
            tmem_ld128(to, r);  // O (the first D columns)
            if (live) {
                if (nsplit_b == 1) {
                    const float inv = 1.f / l_run;
                    __nv_bfloat16* dst =
                        p.out + ((static_cast<size_t>(b) * p.L + l) * p.Hq + kvh * p.G + g) * D;
#pragma unroll
                    for (int c = 0; c < D; c += 8) {
                        const uint4 v = make_uint4(
                            pack_bf16x2(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv),
                            pack_bf16x2(__uint_as_float(r[c + 2]) * inv, __uint_as_float(r[c + 3]) * inv),
                            pack_bf16x2(__uint_as_float(r[c + 4]) * inv, __uint_as_float(r[c + 5]) * inv),
                            pack_bf16x2(__uint_as_float(r[c + 6]) * inv, __uint_as_float(r[c + 7]) * inv));
                        *reinterpret_cast<uint4*>(dst + c) = v;
                    }
                } else {
                    const size_t prow =
                        ((static_cast<size_t>(split) * p.B + b) * p.Hkv + kvh) *
                            (static_cast<size_t>(p.n_mtiles) * kTile) + m;
                    float* dst = p.ws_o + prow * D;
#pragma unroll
                    for (int c = 0; c < D; c += 4)
                        *reinterpret_cast<float4*>(dst + c) =
                            make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                        __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
                    *reinterpret_cast<float2*>(p.ws_ml + prow * 2) = make_float2(m_run, l_run);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Combines the per-split partials (running max m_s, running sum l_s,
// unnormalised O_s) of sequences that were split: one warp per output row.
// Launched as a programmatic dependent of the attention grid: the row's place
// and its number of splits come from ctx_len alone, before waiting for that
// grid; after the wait the splits are read in one pass, four at a time, with
// an online rescale to the running maximum.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnSplitParams p) {
    constexpr int kPer = D / 32;  // columns per lane
    const long gw = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long rows_bk = static_cast<long>(p.G) * p.L;
    const bool valid = gw < rows_bk * p.B * p.Hkv;
    const int m = valid ? static_cast<int>(gw % rows_bk) : 0;
    const int bk = valid ? static_cast<int>(gw / rows_bk) : 0;
    const int kvh = bk % p.Hkv, b = bk / p.Hkv;
    int ns = 0;
    if (valid) {
        int C = p.ctx_group ? (b % p.ctx_group) * p.L : p.ctx_len[b];
        C = C < 0 ? 0 : (C > p.ctx_cap ? p.ctx_cap : C);
        const int nt = (C + kTile - 1) / kTile + p.nblk;
        ns = (nt + p.chunk - 1) / p.chunk;
    }
    // Wait until the attention grid has completed and its partials are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ns <= 1) return;  // not split: written directly by the attention kernel
    const size_t mpad = static_cast<size_t>(p.n_mtiles) * kTile;
    const size_t split_stride = static_cast<size_t>(p.B) * p.Hkv * mpad;
    const size_t base = (static_cast<size_t>(b) * p.Hkv + kvh) * mpad + m;
    float mx = -INFINITY, den = 0.f, acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 4) {
        float pm[4], pl[4], pv[4][kPer];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            pm[u] = -INFINITY;
            pl[u] = 0.f;
#pragma unroll
            for (int j = 0; j < kPer; ++j) pv[u][j] = 0.f;
            if (s0 + u < ns) {
                const size_t r = (s0 + u) * split_stride + base;
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + r * 2));
                pm[u] = ml.x;
                pl[u] = ml.y;
                const float* o = p.ws_o + r * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(o));
                    pv[u][0] = v.x; pv[u][1] = v.y; pv[u][2] = v.z; pv[u][3] = v.w;
                } else {
                    const float2 v = __ldcg(reinterpret_cast<const float2*>(o));
                    pv[u][0] = v.x; pv[u][1] = v.y;
                }
            }
        }
        const float nm = fmaxf(fmaxf(mx, fmaxf(pm[0], pm[1])), fmaxf(pm[2], pm[3]));
        const float sc = ex2_approx(mx - nm);  // 0 on the first round (mx = -inf)
        den *= sc;
#pragma unroll
        for (int j = 0; j < kPer; ++j) acc[j] *= sc;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = ex2_approx(pm[u] - nm);  // 0 for the padding splits
            den += w * pl[u];
#pragma unroll
            for (int j = 0; j < kPer; ++j) acc[j] += w * pv[u][j];
        }
        mx = nm;
    }
    const float inv = 1.f / den;
    const int l = m / p.G, g = m % p.G;
    __nv_bfloat16* dst = p.out + ((static_cast<size_t>(b) * p.L + l) * p.Hq + kvh * p.G + g) * D +
                         lane * kPer;
    if constexpr (kPer == 4) {
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

template <int D>
cudaError_t launch_split_impl(const AttnMaps& m, const AttnSplitParams& p, int splits, cudaStream_t s) {
    dim3 grid(p.n_pairs * splits, p.Hkv, p.B);
    block_attn_split_kernel<D><<<grid, 320, SplitLayout<D>::kAlloc, s>>>(m.q, m.k_ctx, m.v_ctx, m.k_blk,
                                                                  m.v_blk, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_attn_split_kernels() {
    cudaError_t e = cudaFuncSetAttribute(block_attn_split_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SplitLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(block_attn_split_kernel<128>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SplitLayout<128>::kAlloc);
}

cudaError_t launch_block_attn_split(const AttnMaps& maps, const AttnSplitParams& p, int D, int splits,
                                    cudaStream_t s) {
    return D == 64 ? launch_split_impl<64>(maps, p, splits, s) : launch_split_impl<128>(maps, p, splits, s);
}

cudaError_t launch_attn_merge(const AttnSplitParams& p, int D, cudaStream_t s) {
    const long warps = static_cast<long>(p.G) * p.L * p.B * p.Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((warps * 32 + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return D == 64 ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<64>, p)
                   : cudaLaunchKernelEx(&cfg, attn_merge_kernel<128>, p);
}

}  // namespace tt
