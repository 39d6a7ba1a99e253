// Block attention of the TwoTower denoiser ("Nemotron-Labs-TwoTower",
// Section 2.1, Eq. 1): every query of the L-token noisy block takes one
// softmax over [context-tower keys 0..ctx_len-1 of this layer; the block's own
// L keys], with no mask inside the block and GQA head sharing.
//
// One CTA owns one work unit (sequence b, KV head, 128-row query tile, KV
// split). The G = Hq/Hkv query heads of a KV head are packed with the block
// positions into the M dimension (row = l*G + g), so a K/V tile staged once in
// shared memory feeds all of them.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: one query row per thread, reads S from TMEM, online
//              softmax in fp32 (log2 domain), writes P (bf16) to shared memory,
//              rescales O in TMEM when the running max grows by > 2^8
//   warp 4     TMA producer: Q tile once, then K/V tiles into a 2-stage ring
//   warp 5     MMA issuer: S = Q K^T and O += P V on tcgen05 (fp32 in TMEM);
//              owns the TMEM allocation
// TMEM columns: S double buffer at 0 and 128, O at 256 (D columns).
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

constexpr int kStages = 2;
constexpr float kRescaleThresh = 8.0f;  // log2 units

template <int D>
struct AttnLayout {
    static constexpr int kTileBytes = kTile * D * 2;     // a Q, K or V tile (bf16)
    static constexpr int kAtomBytes = kTile * 128;       // one 64-column swizzle atom column
    static constexpr int kPBytes = kTile * kTile * 2;    // a P tile (bf16)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTileBytes;
    static constexpr int kV = kK + kStages * kTileBytes;
    static constexpr int kP = kV + kStages * kTileBytes;
    static constexpr int kBar = kP + 2 * kPBytes;
    // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], pv_done[2], drain
    static constexpr int kNumBars = 1 + 4 * kStages + 7;
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
__global__ void __launch_bounds__(192, 1)
    block_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kc,
                      const __grid_constant__ CUtensorMap tm_vc,
                      const __grid_constant__ CUtensorMap tm_kb,
                      const __grid_constant__ CUtensorMap tm_vb, const AttnParams p) {
    using Lay = AttnLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtile = blockIdx.x % p.n_mtiles;
    const int split = blockIdx.x / p.n_mtiles;
    const int kvh = blockIdx.y, b = blockIdx.z;

    int C = p.ctx_len[b];
    if (C < 0 || C > p.ctx_cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) atomicOr(p.status, kDevCtxLenRange);
        C = C < 0 ? 0 : p.ctx_cap;
    }
    const int nc = (C + kTile - 1) / kTile;
    const int nt = nc + p.nblk;
    const int t0 = split * p.chunk;
    if (t0 >= nt) return;  // this split is past the end of sequence b's keys
    const int n = min(nt, t0 + p.chunk) - t0;
    const int nsplit_b = (nt + p.chunk - 1) / p.chunk;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::kBar);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + kStages;
    uint64_t* v_full = k_empty + kStages;
    uint64_t* v_empty = v_full + kStages;
    uint64_t* s_full = v_empty + kStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = p_full + 2;
    uint64_t* drain = pv_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 128);
            mbar_init(&pv_done[s], 1);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t limit = p.timeout_ns;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_kc);
            tma_prefetch_desc(&tm_vc);
            tma_prefetch_desc(&tm_kb);
            tma_prefetch_desc(&tm_vb);
            bool ok = true;
            uint8_t* sq = sm + Lay::kQ;
            mbar_arrive_expect_tx(q_full, Lay::kTileBytes);
            const int l0 = mtile * (kTile / p.G);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_5d(sq + c * Lay::kAtomBytes, &tm_q, q_full, c * 64, 0, kvh, l0, b);
            int k_issued = 0, v_issued = 0;
            for (int i = 0; i < n; ++i) {
                const int st = i % kStages;
                const uint32_t ph = (i / kStages) & 1;
                const KvTile t = kv_tile(t0 + i, nc, C, p.L);
                if (i >= kStages && !mbar_wait(&k_empty[st], ph ^ 1, limit)) { ok = false; break; }
                uint8_t* sk = sm + Lay::kK + st * Lay::kTileBytes;
                mbar_arrive_expect_tx(&k_full[st], Lay::kTileBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if (t.is_ctx)
                        tma_load_3d(sk + c * Lay::kAtomBytes, &tm_kc, &k_full[st], c * 64, t.base,
                                    b * p.Hkv + kvh);
                    else
                        tma_load_4d(sk + c * Lay::kAtomBytes, &tm_kb, &k_full[st], c * 64, kvh,
                                    t.base, b);
                }
                k_issued = i + 1;
                if (i >= kStages && !mbar_wait(&v_empty[st], ph ^ 1, limit)) { ok = false; break; }
                uint8_t* sv = sm + Lay::kV + st * Lay::kTileBytes;
                mbar_arrive_expect_tx(&v_full[st], Lay::kTileBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if (t.is_ctx)
                        tma_load_3d(sv + c * Lay::kAtomBytes, &tm_vc, &v_full[st], c * 64, t.base,
                                    b * p.Hkv + kvh);
                    else
                        tma_load_4d(sv + c * Lay::kAtomBytes, &tm_vb, &v_full[st], c * 64, kvh,
                                    t.base, b);
                }
                v_issued = i + 1;
            }
            if (!ok) {
                atomicOr(p.status, kDevWaitTimeout);
                // Let the copies already issued land before the CTA can exit.
                mbar_wait(q_full, 0, limit);
                for (int i = k_issued - kStages < 0 ? 0 : k_issued - kStages; i < k_issued; ++i)
                    mbar_wait(&k_full[i % kStages], (i / kStages) & 1, limit);
                for (int i = v_issued - kStages < 0 ? 0 : v_issued - kStages; i < v_issued; ++i)
                    mbar_wait(&v_full[i % kStages], (i / kStages) & 1, limit);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16(kTile, kTile, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, 0, 1);
        bool ok = mbar_wait(q_full, 0, limit);
        const uint32_t sq = smem_u32(sm + Lay::kQ);
        for (int i = 0; i <= n && ok; ++i) {
            if (i < n) {
                const int st = i % kStages;
                if (!mbar_wait(&k_full[st], (i / kStages) & 1, limit)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sk = smem_u32(sm + Lay::kK + st * Lay::kTileBytes);
                    const uint32_t d_s = tmem + (i & 1) * kTile;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * Lay::kAtomBytes + (kk & 3) * 32;
                        tc_mma_ss(d_s, sdesc_sw128(sq + off, 16, 1024),
                                  sdesc_sw128(sk + off, 16, 1024), idesc_qk, kk > 0);
                    }
                    tc_commit(&s_full[i & 1]);
                    tc_commit(&k_empty[st]);
                }
                __syncwarp();
            }
            if (i >= 1) {
                const int t = i - 1;
                const int pb = t & 1, vs = t % kStages;
                if (!mbar_wait(&p_full[pb], (t >> 1) & 1, limit) ||
                    !mbar_wait(&v_full[vs], (t / kStages) & 1, limit)) {
                    ok = false;
                    break;
                }
                const KvTile kt = kv_tile(t0 + t, nc, C, p.L);
                if (kt.is_ctx && kt.valid < kTile) {
                    // Cache rows past ctx_len may hold anything (even NaN);
                    // P is 0 there, but 0 * NaN is not, so zero those V rows.
                    uint8_t* sv = sm + Lay::kV + vs * Lay::kTileBytes;
                    const int rows = kTile - kt.valid;
                    for (int u = lane; u < rows * 8 * (D / 64); u += 32) {
                        const int c = u / (rows * 8);
                        const int rem = u % (rows * 8);
                        const int r = kt.valid + rem / 8;
                        *reinterpret_cast<uint4*>(sv + c * Lay::kAtomBytes + r * 128 +
                                                  (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sp = smem_u32(sm + Lay::kP + pb * Lay::kPBytes);
                    const uint32_t sv = smem_u32(sm + Lay::kV + vs * Lay::kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t ad =
                            sdesc_sw128(sp + (kk >> 2) * Lay::kAtomBytes + (kk & 3) * 32, 16, 1024);
                        // V is MN-major (d contiguous): 16 keys = two 8-row atoms;
                        // the next 64 columns of d sit one atom column further.
                        const uint64_t bd = sdesc_sw128(sv + kk * 2048, Lay::kAtomBytes, 1024);
                        tc_mma_ss(tmem + 2 * kTile, ad, bd, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&pv_done[pb]);
                    tc_commit(&v_empty[vs]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        // No MMA may still be running when the TMEM is released.
        if (lane == 0) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, limit);
    } else {
        // ------------------------------------------------------------ softmax
        const int row = warp * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int sb = i & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (i >> 1) & 1, limit));
            if (!ok) break;
            tc_fence_after();
            float s[kTile];
#pragma unroll
            for (int c4 = 0; c4 < kTile / 32; ++c4) {
                uint32_t r[32];
                tmem_ld32(tl + sb * kTile + c4 * 32, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) s[c4 * 32 + j] = __uint_as_float(r[j]);
            }
            const KvTile kt = kv_tile(t0 + i, nc, C, p.L);
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTile; ++c) {
                s[c] = (c < kt.valid) ? s[c] : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            const float m_tile = mx * sl2;
            if (i == 0) {
                m_run = m_tile;
            } else if (m_tile > m_run + kRescaleThresh) {
                const float alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
                l_run *= alpha;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, limit));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t r[32];
                    tmem_ld32(tl + 2 * kTile + c4 * 32, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                    tmem_st32(tl + 2 * kTile + c4 * 32, r);
                }
            }
            if (i >= 2) {
                ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[sb], ((i - 2) >> 1) & 1, limit));
                if (!ok) break;
            }
            uint8_t* pbuf = sm + Lay::kP + sb * Lay::kPBytes + row * 128;
            const float neg_m = -m_run;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    float e[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        e[x] = ex2_approx(fmaf(s[c * 64 + u * 8 + x], sl2, neg_m));
                        lsum += e[x];
                    }
                    const uint4 v = make_uint4(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]),
                                               pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
                    *reinterpret_cast<uint4*>(pbuf + c * Lay::kAtomBytes + ((u ^ (row & 7)) << 4)) = v;
                }
            }
            l_run += lsum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[sb]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, limit));
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kDevWaitTimeout);
        } else {
            tc_fence_after();
            const int m = mtile * kTile + row;
            const int l = m / p.G, g = m % p.G;
            const bool live = l < p.L;
            if (nsplit_b == 1) {
                const float inv = 1.f / l_run;
                __nv_bfloat16* dst =
                    p.out + ((static_cast<size_t>(b) * p.L + l) * p.Hq + kvh * p.G + g) * D;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t r[32];
                    tmem_ld32(tl + 2 * kTile + c4 * 32, r);
                    if (live) {
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            const uint4 v = make_uint4(
                                pack_bf16x2(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv),
                                pack_bf16x2(__uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv),
                                pack_bf16x2(__uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv),
                                pack_bf16x2(__uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv));
                            *reinterpret_cast<uint4*>(dst + c4 * 32 + j) = v;
                        }
                    }
                }
            } else {
                const size_t prow =
                    ((static_cast<size_t>(split) * p.B + b) * p.Hkv + kvh) *
                        (static_cast<size_t>(p.n_mtiles) * kTile) + m;
                float* dst = p.ws_o + prow * D;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t r[32];
                    tmem_ld32(tl + 2 * kTile + c4 * 32, r);
                    if (live) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + c4 * 32 + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    }
                }
                if (live) *reinterpret_cast<float2*>(p.ws_ml + prow * 2) = make_float2(m_run, l_run);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Combines the per-split partials (running max m_s, running sum l_s,
// unnormalised O_s) of sequences that were split: one warp per output row.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnParams p) {
    constexpr int kPer = D / 32;  // columns per lane
    const long gw = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long rows_bk = static_cast<long>(p.G) * p.L;
    if (gw >= rows_bk * p.B * p.Hkv) return;
    const int m = static_cast<int>(gw % rows_bk);
    const int bk = static_cast<int>(gw / rows_bk);
    const int kvh = bk % p.Hkv, b = bk / p.Hkv;
    int C = p.ctx_len[b];
    C = C < 0 ? 0 : (C > p.ctx_cap ? p.ctx_cap : C);
    const int nt = (C + kTile - 1) / kTile + p.nblk;
    const int ns = (nt + p.chunk - 1) / p.chunk;
    if (ns == 1) return;  // written directly by the attention kernel
    const size_t mpad = static_cast<size_t>(p.n_mtiles) * kTile;
    const size_t split_stride = static_cast<size_t>(p.B) * p.Hkv * mpad;
    const size_t base = (static_cast<size_t>(b) * p.Hkv + kvh) * mpad + m;
    float mx = -INFINITY;
    for (int s = 0; s < ns; ++s) mx = fmaxf(mx, p.ws_ml[(s * split_stride + base) * 2]);
    float den = 0.f, acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + (s * split_stride + base) * 2);
        const float w = ex2_approx(ml.x - mx);
        den += w * ml.y;
        const float* o = p.ws_o + (s * split_stride + base) * D + lane * kPer;
        if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4*>(o);
            acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(o);
            acc[0] += w * v.x; acc[1] += w * v.y;
        }
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
cudaError_t launch_attn_impl(const AttnMaps& m, const AttnParams& p, int splits, cudaStream_t s) {
    dim3 grid(p.n_mtiles * splits, p.Hkv, p.B);
    block_attn_kernel<D><<<grid, 192, AttnLayout<D>::kAlloc, s>>>(m.q, m.k_ctx, m.v_ctx, m.k_blk,
                                                                  m.v_blk, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_attn_kernels() {
    cudaError_t e = cudaFuncSetAttribute(block_attn_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         AttnLayout<64>::kAlloc);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(block_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnLayout<128>::kAlloc);
}

int attn_smem_bytes(int D) {
    return D == 64 ? AttnLayout<64>::kAlloc : AttnLayout<128>::kAlloc;
}

cudaError_t launch_block_attn(const AttnMaps& maps, const AttnParams& p, int D, int splits,
                              cudaStream_t s) {
    return D == 64 ? launch_attn_impl<64>(maps, p, splits, s)
                   : launch_attn_impl<128>(maps, p, splits, s);
}

cudaError_t launch_attn_merge(const AttnParams& p, int D, cudaStream_t s) {
    const long warps = static_cast<long>(p.G) * p.L * p.B * p.Hkv;
    const unsigned blocks = static_cast<unsigned>((warps * 32 + 255) / 256);
    if (D == 64)
        attn_merge_kernel<64><<<blocks, 256, 0, s>>>(p);
    else
        attn_merge_kernel<128><<<blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tt
