// The denoiser's LM head with the commit step behind it ("Nemotron-Labs-
// TwoTower", Section 2.2, Algorithm 2: the denoiser's distribution over the
// vocabulary for every position of the block, then ConfidenceSample on it).
//
// lm_head_kernel: logits[M][V] = hidden[M][K] * W[V][K]^T in fp32 from bf16
// operands on the tensor core (tcgen05, accumulators in TMEM). Its epilogue,
// which reads every logit once anyway, also folds each row's maximum and first
// argmax into one 64-bit word per row (an atomic max of an order-preserving
// (value, -index) encoding), so the commit step needs no pass of its own for
// them.
//   Persistent: one CTA per SM walks 128 x 256 output tiles in vocabulary-block
//   order (the CTAs running at the same time share a block of W through L2;
//   hidden stays in L2). Warp 0: TMA producer (A 128x64 and B 256x64 bf16
//   tiles, 128-byte swizzle, a 4-stage ring); warp 1: MMA issuer (M=128,
//   N=256, K=16 steps) and TMEM owner, two 256-column accumulators so that
//   the epilogue of a tile overlaps the MMAs of the next; warps 2-5: epilogue
//   (TMEM lane quarter = warp % 4), 32 columns at a time.
//
// commit_rowmax_kernel: the commit step given each row's maximum and
// prediction. A masked row's canonical key is a sum of fixed-point terms over
// its logits; with the maximum known, any chunk of a row can be summed on any
// SM and the partial sums added with 64-bit integer atomics (the total does
// not depend on the order). The work is (row, 8192-logit chunk) units in
// row-major order, one contiguous range per CTA (one CTA per SM): a producer
// warp streams the masked rows' chunks through a 3-slot shared-memory ring of
// 64 KB bulk copies, 16 warps sum the terms (4 per scheduler, enough to keep
// the FMA pipe fed; fewer or smaller chunks measured slower); a row's partial key stays in
// registers until the row ends, then one atomic add; each CTA counts its units
// of a block on the block's ticket once, and the CTA that completes the count
// (L * chunks per row) ranks the block's masked rows and commits. Every row's
// mask is read before it is counted, so the mask may be updated in place.
#include "commit_key.cuh"
#include "commit_select.cuh"
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kAStage = kBM * kBK * 2;           // 16 KB
constexpr int kBStage = kBN * kBK * 2;           // 32 KB
constexpr int kStageBytes = kAStage + kBStage;
constexpr int kGemmThreads = 192;
constexpr int kBarOff = kStages * kStageBytes;   // full[4], empty[4], acc_full[2], acc_empty[2], drain
constexpr int kTmemSlotOff = kBarOff + (2 * kStages + 5) * 8;
constexpr int kGemmSmem = kTmemSlotOff + 16 + 1024;

__device__ __forceinline__ unsigned long long atom_max_u64(unsigned long long* a, unsigned long long v) {
    return atomicMax(a, v);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const LmHeadParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kBarOff);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kTmemSlotOff);

    const int mt = (p.M + kBM - 1) / kBM, nt = (p.V + kBN - 1) / kBN;
    const long long tiles = static_cast<long long>(mt) * nt;
    const int ksteps = (p.K + kBK - 1) / kBK;
    const uint64_t limit = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 128);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
            bool ok = true;
            int li = 0;  // stage loads issued
            for (long long t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int m0 = static_cast<int>(t % mt) * kBM, n0 = static_cast<int>(t / mt) * kBN;
                for (int ks = 0; ks < ksteps; ++ks, ++li) {
                    const int s = li % kStages;
                    if (li >= kStages && !mbar_wait(&empty[s], ((li / kStages) & 1) ^ 1, limit)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = sm + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    tma_load_2d(st, &tm_a, &full[s], ks * kBK, m0);
                    tma_load_2d(st + kAStage, &tm_b, &full[s], ks * kBK, n0);
                }
            }
            if (!ok) atomicOr(p.status, kDevWaitTimeout);
            // the copies in flight land before the CTA can leave
            const uint64_t dl = drain_limit(limit);
            for (int l = li - kStages < 0 ? 0 : li - kStages; l < li; ++l)
                mbar_wait(&full[l % kStages], (l / kStages) & 1, dl);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_bf16(kBM, kBN, 0, 0);
        const uint32_t base = smem_u32(sm);
        bool ok = true;
        int li = 0, nt_local = 0;
        for (long long t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++nt_local) {
            const int buf = nt_local & 1;
            // the epilogue has read this accumulator's previous tile
            if (nt_local >= 2 && !mbar_wait(&acc_empty[buf], ((nt_local >> 1) - 1) & 1, limit)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int ks = 0; ks < ksteps; ++ks, ++li) {
                const int s = li % kStages;
                if (!mbar_wait(&full[s], (li / kStages) & 1, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kAStage;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_ss(tmem + buf * kBN, sdesc_sw128(sa + kk * 32, 16, 1024),
                                  sdesc_sw128(sb + kk * 32, 16, 1024), idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) tc_commit(&acc_full[buf]);
            __syncwarp();
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        if (lane == 0) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, drain_limit(limit));
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        int nt_local = 0;
        for (long long t = blockIdx.x; t < tiles; t += gridDim.x, ++nt_local) {
            const int buf = nt_local & 1;
            const int m0 = static_cast<int>(t % mt) * kBM, n0 = static_cast<int>(t / mt) * kBN;
            ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (nt_local >> 1) & 1, limit));
            if (!ok) break;
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            float best = -INFINITY;
            int bcol = 0;
            float* dst = p.logits + static_cast<size_t>(row) * p.V + n0;
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + buf * kBN + c * 32, r);
                const int col0 = n0 + c * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float v = __uint_as_float(r[j]);
                    if (col0 + j < p.V && v > best) {
                        best = v;
                        bcol = col0 + j;
                    }
                }
                if (row < p.M) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        if (col0 + j < p.V)
                            *reinterpret_cast<float4*>(dst + c * 32 + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[buf]);
            if (row < p.M && best > -INFINITY) atom_max_u64(p.rowmax + row, key::enc_argmax(best, bcol));
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- commit given the row maximum
constexpr int kTermConsumers = 512;                     // warps 1-16: the term sums
constexpr int kTermThreads = 32 + kTermConsumers;       // warp 0: the producer
constexpr int kTermChunk = 16384;                       // logits per unit (64 KB)
constexpr int kTermSlots = 3;                           // ring depth
constexpr int kTermPer = kTermChunk / kTermConsumers;   // 32 per consumer thread
constexpr int kTermBarOff = kTermSlots * kTermChunk * 4;
constexpr int kTermSmem = kTermBarOff + 2 * kTermSlots * 8 + 1024;

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* a, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}

// Barrier among the consumer warps only (id 1; 0 is __syncthreads).
__device__ __forceinline__ void consumers_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kTermConsumers) : "memory");
}

__global__ void __launch_bounds__(kTermThreads, 1)
    commit_rowmax_kernel(const RowmaxCommitParams p) {
    extern __shared__ uint8_t term_smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(term_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* ring = reinterpret_cast<float*>(sm);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kTermBarOff);
    uint64_t* empty = full + kTermSlots;
    __shared__ unsigned long long s_part[kTermConsumers / 32];
    __shared__ int s_last;
    __shared__ unsigned long long s_key[sel::kSelChunk];
    __shared__ uint32_t s_mbits[kCommitMaxL / 32], s_cbits[kCommitMaxL / 32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (p.V + kTermChunk - 1) / kTermChunk;
    const long long units = static_cast<long long>(p.B) * p.L * nch;
    const unsigned per_block = static_cast<unsigned>(p.L) * nch;
    // this CTA's contiguous range of units (row-major): a row's chunks follow
    // one another, so its partial key stays in registers until the row ends
    const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    const uint64_t limit = p.timeout_ns;
    if (tid == 0) {
        for (int i = 0; i < kTermSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kTermConsumers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Bulk copies of the masked rows' chunks (L2 evict-first) into the ring,
        // in unit order; a row's mask is read here before its units are counted
        // on the block's ticket by the consumers.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int it = 0;
            bool ok = true;
            int r = static_cast<int>(u0 / nch), c = static_cast<int>(u0 % nch);
            bool cur_masked = u0 < u1 && __ldcg(p.masked + r) != 0;
            for (long long u = u0; u < u1 && ok; ++u, ++c) {
                if (c == nch) {
                    c = 0;
                    ++r;
                    cur_masked = __ldcg(p.masked + r) != 0;
                }
                if (!cur_masked) continue;
                const int s = it % kTermSlots;
                if (it >= kTermSlots && !mbar_wait(&empty[s], ((it / kTermSlots) - 1) & 1, limit)) {
                    ok = false;
                    break;
                }
                const int v0 = c * kTermChunk, n = min(kTermChunk, p.V - v0);
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(n) * 4);
                bulk_load(ring + static_cast<size_t>(s) * kTermChunk,
                          p.logits + static_cast<size_t>(r) * p.V + v0, static_cast<uint32_t>(n) * 4,
                          &full[s], pol);
                ++it;
            }
            if (!ok) atomicOr(p.status, kDevWaitTimeout);
            // the copies issued last land before the CTA can exit
            const uint64_t dl = drain_limit(limit);
            for (int j = it - kTermSlots < 0 ? 0 : it - kTermSlots; j < it; ++j)
                mbar_wait(&full[j % kTermSlots], (j / kTermSlots) & 1, dl);
        }
        __syncwarp();
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int ct = tid - 32;  // consumer thread
    const int cw = warp - 1;  // consumer warp
    int cur_r = -1, cur_b = -1;
    bool cur_masked = false, ok = true;
    key::f2 m2 = 0;
    unsigned hi = 0, lo = 0;
    int cnt = 0;
    unsigned bunits = 0;  // this CTA's units of block cur_b
    int it = 0;

    // adds the CTA's partial key of row cur_r to key[cur_r]
    auto flush_row = [&]() {
        if (cur_r < 0 || !cur_masked) return;
        hi -= static_cast<unsigned>(cnt) * key::kMagic43Bits;
        lo -= static_cast<unsigned>(cnt) * key::kMagic23Bits;
        unsigned long long acc = (static_cast<unsigned long long>(hi) << 20) +
                                 static_cast<long long>(static_cast<int>(lo));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s_part[cw] = acc;
        consumers_bar();
        if (ct == 0) {
            unsigned long long tot = 0;
#pragma unroll
            for (int w = 0; w < kTermConsumers / 32; ++w) tot += s_part[w];
            atomicAdd(p.key + cur_r, tot);
        }
        consumers_bar();
        hi = lo = 0;
        cnt = 0;
    };
    // counts this CTA's units of block cur_b; the CTA that completes the
    // block's count ranks it and commits
    auto flush_block = [&]() {
        if (cur_b < 0) return;
        if (ct == 0) {
            __threadfence();  // this CTA's key additions before its ticket
            const unsigned t = atom_add_acq_rel(p.blk + cur_b, bunits);
            s_last = t + bunits == per_block;
            if (s_last) p.blk[cur_b] = 0;  // no other ticket of this call remains
        }
        consumers_bar();
        if (s_last && cw == 0) {
            __threadfence();
            const size_t base = static_cast<size_t>(cur_b) * p.L;
            int n = 0;
            for (int i = lane; i < p.L; i += 32) {
                const bool mi = __ldcg(p.masked + base + i) != 0;
                n += mi;
                if (mi) p.arg[base + i] = key::dec_index(__ldcg(p.rowmax + base + i));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
            __syncwarp();
            if (p.L <= 32 * sel::kSelRegRows) sel::select_block_small(p, cur_b, n, lane);
            else sel::select_block(p, cur_b, n, s_key, s_mbits, s_cbits, lane);
            // keys out for tt_commit_keys; the block's accumulators back to zero
            for (int i = lane; i < p.L; i += 32) {
                p.key_out[base + i] = __ldcg(p.key + base + i);
                p.key[base + i] = 0ull;
                p.rowmax[base + i] = 0ull;
            }
        }
        consumers_bar();
        bunits = 0;
    };

    int r = static_cast<int>(u0 / nch), c = static_cast<int>(u0 % nch) - 1;
    for (long long u = u0; u < u1; ++u) {
        if (++c == nch) {
            c = 0;
            ++r;
        }
        if (r != cur_r) {
            flush_row();
            const int b = r / p.L;
            if (b != cur_b) {
                flush_block();
                cur_b = b;
            }
            cur_r = r;
            // the row's mask is read before this CTA counts it on the block's ticket
            cur_masked = __ldcg(p.masked + r) != 0;
            if (!cur_masked && ct == 0 && c == 0) p.masked_out[r] = 0;  // the selection writes masked rows
            if (cur_masked) m2 = key::dup(key::dec_value(__ldcg(p.rowmax + r)));
        }
        ++bunits;
        if (!cur_masked || !ok) continue;
        const int s = it % kTermSlots;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (it / kTermSlots) & 1, limit));
        ++it;
        if (!ok) continue;  // keeps counting the units so that no ticket wait can hang
        const int n = min(kTermChunk, p.V - c * kTermChunk);
        const float4* src = reinterpret_cast<const float4*>(ring + static_cast<size_t>(s) * kTermChunk);
        float4 x[kTermPer / 4];
#pragma unroll
        for (int j = 0; j < kTermPer / 4; ++j) x[j] = src[j * kTermConsumers + ct];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp has read its part of the slot
#pragma unroll
        for (int j = 0; j < kTermPer / 4; ++j) {
            if (4 * (j * kTermConsumers + ct) >= n) continue;
            float d0, d1, d2, d3;
            key::upk(key::fsub2(key::pk(x[j].x, x[j].y), m2), d0, d1);
            key::upk(key::fsub2(key::pk(x[j].z, x[j].w), m2), d2, d3);
            // differences below -31 have term 0; clamped there (keeps n and the
            // exponent arithmetic in range)
            key::add_terms(key::pk(fmaxf(d0, -31.0f), fmaxf(d1, -31.0f)), hi, lo);
            key::add_terms(key::pk(fmaxf(d2, -31.0f), fmaxf(d3, -31.0f)), hi, lo);
            cnt += 4;
        }
    }
    if (!ok && ct == 0) atomicOr(p.status, kDevWaitTimeout);
    flush_row();
    flush_block();
}

}  // namespace

size_t lm_head_smem_bytes() { return kGemmSmem; }

cudaError_t configure_lm_head_kernels() {
    const cudaError_t e =
        cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(commit_rowmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTermSmem);
}

cudaError_t launch_lm_head(const CUtensorMap& a, const CUtensorMap& b, const LmHeadParams& p, int num_sms,
                           cudaStream_t s) {
    const long long tiles = static_cast<long long>((p.M + kBM - 1) / kBM) * ((p.V + kBN - 1) / kBN);
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    lm_head_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(a, b, p);
    return cudaGetLastError();
}

cudaError_t launch_commit_rowmax(const RowmaxCommitParams& p, int num_sms, cudaStream_t s) {
    // one CTA per SM, every CTA's range at once (the ranges are equal)
    const long long units = static_cast<long long>(p.B) * p.L * ((p.V + kTermChunk - 1) / kTermChunk);
    const int grid = static_cast<int>(units < num_sms ? units : num_sms);
    commit_rowmax_kernel<<<grid, kTermThreads, kTermSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tt
