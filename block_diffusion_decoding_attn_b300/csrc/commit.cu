// Unmask/commit step of the TwoTower sampler ("Nemotron-Labs-TwoTower",
// Section 2.2, Algorithm 2, confidence unmasking) with a fixed budget of k
// commits per block per step. One launch:
//
// One 8-CTA cluster per row: each CTA bulk-copies its 1/8 slice of the fp32
// logit row into shared memory (TMA, evict-first) and finds the slice's max
// and first argmax; the cluster agrees on the row maximum m through
// distributed shared memory; each CTA then sums the canonical fixed-point
// terms q(l_v - m) of its slice from shared memory and CTA 0 adds the eight
// partial sums:
//     key[r] = sum_v rint(2^40 * e(RN32(l_v - m))),  arg[r] = first argmax
// The sum is an integer, so the key does not depend on the reduction order and
// matches a scalar CPU loop bit for bit. key / 2^40 = 1 / (max softmax
// probability) up to the rounding of e; smaller key = more confident.
// Every row's cluster then takes a ticket for its block; the cluster that
// takes the last ticket ranks the block's masked rows by (key, row) and
// commits the first min(k, #masked): tok[r] = arg[r], masked_out[r] = 0.
//
// e(x) is an fp32 exponential defined for this purpose (Cody and Waite range
// reduction, then the degree-7 Taylor polynomial of exp, all with
// round-to-nearest fused multiply-adds):
//   x < -30 -> term 0
//   n = nearest integer (ties to even) to the exact product x * log2(e)
//   r = fma(-n, C1, x), r = fma(-n, C2, r)     C1 = RN32(ln 2), C2 = RN32(ln 2 - C1)
//   p = c7; p = fma(p, r, c_j), j = 6..0       c_j = RN32(1 / j!)
//   term = rint(p * 2^(n + 40))
// The term is formed without any float-to-64-bit conversion (those run on the
// FP64 pipe, which is narrow on this part): the polynomial carries the 2^40
// factor in its coefficients (exact power-of-two scaling), 2^n is added to the
// exponent field, and rint splits into a multiple of 2^20 plus a remainder,
// both read out of the bits of exact fp32 sums. The arithmetic runs on packed
// f32x2 pairs (each half rounded exactly like the scalar operation).
#include <cooperative_groups.h>

#include "ptx.cuh"
#include "tt_internal.h"

namespace cg = cooperative_groups;

namespace tt {

namespace {

// RN32(1/ln 2), RN32(ln 2), RN32(ln 2 - RN32(ln 2)); 2^40 * RN32(1/j!)
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e430p-1f;
constexpr float kLn2Lo = -0x1.05c610p-29f;
constexpr float kC0 = 0x1.000000p+40f;
constexpr float kC2 = 0x1.000000p+39f;
constexpr float kC3 = 0x1.555556p+37f;
constexpr float kC4 = 0x1.555556p+35f;
constexpr float kC5 = 0x1.111112p+33f;
constexpr float kC6 = 0x1.6c16c2p+30f;
constexpr float kC7 = 0x1.a01a02p+27f;
constexpr float kMagic23 = 0x1.8p+23f;  // fp32 sums in [2^23, 2^24) have ulp 1
constexpr float kMagic43 = 0x1.8p+43f;  // ... in [2^43, 2^44) have ulp 2^20
constexpr int kMagic23Bits = 0x4B400000;
constexpr int kMagic43Bits = 0x55400000;

// Packed fp32 pairs: one f32x2 instruction does the same round-to-nearest
// operation on both halves, halving the issue slots of the term arithmetic.
using f2 = unsigned long long;

__device__ __forceinline__ f2 pk(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(f2 r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f2 dup(float c) { return pk(c, c); }
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Adds rint(2^40 * e(x0)) + rint(2^40 * e(x1)) (x <= 0) to the pair
// (hi, lo): sum of terms = hi * 2^20 + lo.
__device__ __forceinline__ void add_fixed_terms(float x0, float x1, unsigned& hi, int& lo) {
    const f2 x = pk(fmaxf(x0, -31.0f), fmaxf(x1, -31.0f));  // terms below -30 are 0 either way
    const f2 nb = fma2(x, dup(kLog2e), dup(kMagic23));     // 1.5*2^23 + n
    const f2 n = sub2(nb, dup(kMagic23));
    f2 r = fma2(n, dup(-kLn2Hi), x);
    r = fma2(n, dup(-kLn2Lo), r);
    f2 p = fma2(dup(kC7), r, dup(kC6));
    p = fma2(p, r, dup(kC5));
    p = fma2(p, r, dup(kC4));
    p = fma2(p, r, dup(kC3));
    p = fma2(p, r, dup(kC2));
    p = fma2(p, r, dup(kC0));
    p = fma2(p, r, dup(kC0));  // 2^40 * p(r), in [2^39.5, 2^40.5]
    float p0, p1, nb0, nb1;
    upk(p, p0, p1);
    upk(nb, nb0, nb1);
    // y = p * 2^n: add n to the exponent field; (bits(nb) << 23) == (n << 23) mod 2^32.
    const f2 y = pk(__int_as_float(__float_as_int(p0) + (__float_as_int(nb0) << 23)),
                    __int_as_float(__float_as_int(p1) + (__float_as_int(nb1) << 23)));
    const f2 a = add2(y, dup(kMagic43));               // 1.5*2^43 + 2^20 * round(y / 2^20)
    const f2 rem = sub2(y, sub2(a, dup(kMagic43)));    // exact, |rem| <= 2^19
    const f2 b = add2(rem, dup(kMagic23));             // 1.5*2^23 + rint(rem)
    float a0, a1, b0, b1;
    upk(a, a0, a1);
    upk(b, b0, b1);
    hi += static_cast<unsigned>(__float_as_int(a0) - kMagic43Bits) +
          static_cast<unsigned>(__float_as_int(a1) - kMagic43Bits);
    lo += (__float_as_int(b0) - kMagic23Bits) + (__float_as_int(b1) - kMagic23Bits);
}

struct ArgMax {
    float v;
    int i;
};

// Larger value wins; equal values -> lower index (first occurrence).
__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

constexpr int kPieces = 4;  // bulk copies per slice, each with its own barrier

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Ranks the masked rows of block b by (key, row) and commits the first k.
// Reads go through L2: the keys were written by other SMs.
__device__ void select_block(const CommitParams& p, int b, unsigned long long* s_key,
                             uint8_t* s_m) {
    const size_t base = static_cast<size_t>(b) * p.L;
    for (int i = threadIdx.x; i < p.L; i += blockDim.x) {
        const uint8_t mk = __ldcg(p.masked + base + i);
        s_m[i] = mk;
        s_key[i] = mk ? __ldcg(p.key + base + i) : 0ull;
    }
    __syncthreads();  // every read of masked precedes any write of masked_out (they may alias)
    for (int i = threadIdx.x; i < p.L; i += blockDim.x) {
        if (!s_m[i]) {
            p.masked_out[base + i] = 0;
            continue;
        }
        const unsigned long long ki = s_key[i];
        int rank = 0;
        for (int j = 0; j < p.L; ++j)
            rank += (s_m[j] && (s_key[j] < ki || (s_key[j] == ki && j < i))) ? 1 : 0;
        if (rank < p.k) {
            p.tok[base + i] = __ldcg(p.arg + base + i);
            p.masked_out[base + i] = 0;
        } else {
            p.masked_out[base + i] = 1;
        }
    }
}

__global__ void __cluster_dims__(kCommitCluster, 1, 1) __launch_bounds__(kCommitThreads)
    commit_kernel(const CommitParams p) {
    extern __shared__ __align__(128) unsigned char dyn[];
    float* slice = reinterpret_cast<float*>(dyn);
    __shared__ __align__(8) uint64_t bars[kPieces];
    __shared__ ArgMax red_am[kCommitThreads / 32];
    __shared__ unsigned long long red_s[kCommitThreads / 32];
    __shared__ ArgMax cta_am;               // this CTA's (max, argmax), read by the cluster
    __shared__ unsigned long long cta_sum;  // this CTA's partial key, read by rank 0
    __shared__ ArgMax row_am;
    __shared__ int is_last;

    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kCommitCluster;
    const int blk = row / p.L;
    const unsigned rank = cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // uniform over the cluster: all its CTAs read the same flag
    const bool masked = p.masked[row] != 0;

    if (masked) {
        const int v0 = static_cast<int>(rank) * p.slice;
        const int cnt = max(0, min(p.slice, p.V - v0));  // multiple of 4
        const float* src = p.logits + static_cast<size_t>(row) * p.V + v0;
        const int per = (((cnt + kPieces - 1) / kPieces) + 3) & ~3;  // floats per piece

        if (tid == 0) {
            for (int i = 0; i < kPieces; ++i) mbar_init(&bars[i], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            const uint64_t pol = l2_policy_evict_first();
            for (int i = 0; i < kPieces; ++i) {
                const int lo = i * per, hi = min(cnt, lo + per);
                if (hi > lo) {
                    mbar_arrive_expect_tx(&bars[i], (hi - lo) * 4);
                    bulk_load(slice + lo, src + lo, (hi - lo) * 4, &bars[i], pol);
                }
            }
        }

        // Pass 1: slice max, piece by piece as it lands; per thread the first
        // float4 group that reaches its running max is remembered.
        float best = -INFINITY;
        int bestg = -1;
        bool ok = true;
        for (int i = 0; i < kPieces; ++i) {
            const int lo = i * per, hi = min(cnt, lo + per);
            if (hi <= lo) break;
            if (!mbar_wait(&bars[i], 0, p.timeout_ns)) { ok = false; break; }
            for (int e = lo + tid * 4; e < hi; e += kCommitThreads * 4) {
                const float4 x = *reinterpret_cast<const float4*>(slice + e);
                const float g = fmaxf(max3(x.x, x.y, x.z), x.w);
                if (g > best) { best = g; bestg = e; }
            }
        }
        if (!ok) {
            if (tid == 0) atomicOr(p.status, kDevWaitTimeout);
            // Let every copy already issued land before this CTA can exit.
            for (int i = 0; i < kPieces; ++i)
                if (min(cnt, i * per + per) > i * per) mbar_wait(&bars[i], 0, p.timeout_ns);
        }
        ArgMax am{-INFINITY, 0x7fffffff};
        if (ok && bestg >= 0) {
            const float4 x = *reinterpret_cast<const float4*>(slice + bestg);
            const int j = x.x == best ? 0 : x.y == best ? 1 : x.z == best ? 2 : 3;
            am = ArgMax{best, v0 + bestg + j};
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ArgMax other{__shfl_xor_sync(0xffffffffu, am.v, o),
                         __shfl_xor_sync(0xffffffffu, am.i, o)};
            am = better(am, other);
        }
        if (lane == 0) red_am[warp] = am;
        __syncthreads();
        if (tid == 0) {
            ArgMax a = red_am[0];
            for (int w = 1; w < kCommitThreads / 32; ++w) a = better(a, red_am[w]);
            cta_am = a;
        }
        cluster.sync();
        if (tid == 0) {
            ArgMax a{-INFINITY, 0x7fffffff};
            for (int r = 0; r < kCommitCluster; ++r)
                a = better(a, *cluster.map_shared_rank(&cta_am, r));
            row_am = a;
        }
        __syncthreads();
        const float m = row_am.v;

        // Pass 2: fixed-point confidence terms of the slice.
        unsigned hi = 0;
        int lo = 0;
        if (ok) {
            for (int e = tid * 4; e < cnt; e += kCommitThreads * 4) {
                const float4 x = *reinterpret_cast<const float4*>(slice + e);
                float d0, d1, d2, d3;
                upk(sub2(pk(x.x, x.y), dup(m)), d0, d1);
                upk(sub2(pk(x.z, x.w), dup(m)), d2, d3);
                add_fixed_terms(d0, d1, hi, lo);
                add_fixed_terms(d2, d3, hi, lo);
            }
        }
        unsigned long long acc =
            (static_cast<unsigned long long>(hi) << 20) + static_cast<long long>(lo);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) red_s[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            unsigned long long s = 0;
            for (int w = 0; w < kCommitThreads / 32; ++w) s += red_s[w];
            cta_sum = s;
        }
        cluster.sync();
        if (rank == 0 && tid == 0) {
            unsigned long long s = 0;
            for (int r = 0; r < kCommitCluster; ++r) s += *cluster.map_shared_rank(&cta_sum, r);
            p.key[row] = s;
            p.arg[row] = row_am.i;
        }
        cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
    }
    if (rank != 0) return;

    // Block ticket: the cluster of the block's last row to finish commits.
    if (tid == 0) {
        __threadfence();  // this row's key/arg before the ticket
        const unsigned t = atomicInc(p.counters + blk, static_cast<unsigned>(p.L - 1));
        is_last = t == static_cast<unsigned>(p.L - 1);  // the counter wrapped back to 0
        __threadfence();
    }
    __syncthreads();
    if (!is_last) return;
    select_block(p, blk, reinterpret_cast<unsigned long long*>(dyn),
                 dyn + static_cast<size_t>(p.L) * 8);
}

}  // namespace

size_t commit_smem_bytes(int V, int L) {
    const size_t slice = static_cast<size_t>((((V + kCommitCluster - 1) / kCommitCluster) + 3) & ~3) * 4;
    const size_t sel = static_cast<size_t>(L) * 9;
    return slice > sel ? slice : sel;
}

cudaError_t launch_commit(const CommitParams& p, cudaStream_t s) {
    commit_kernel<<<static_cast<unsigned>(p.B * p.L) * kCommitCluster, kCommitThreads,
                    commit_smem_bytes(p.V, p.L), s>>>(p);
    return cudaGetLastError();
}

cudaError_t configure_commit_kernels() {
    return cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCommitSmemMax);
}

}  // namespace tt
