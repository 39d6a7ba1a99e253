// Unmask/commit step of the TwoTower sampler ("Nemotron-Labs-TwoTower",
// Section 2.2, Algorithm 2, confidence unmasking) with a fixed budget of k
// commits per block per step.
//
// Kernel 1 (commit_rows_kernel), one 8-CTA cluster per still-masked row:
//   each CTA bulk-copies its 1/8 slice of the fp32 logit row into shared
//   memory (TMA, evict-first), finds max / first argmax, the cluster agrees
//   on the row maximum m through distributed shared memory, then each CTA
//   sums the canonical fixed-point terms q(l_v - m) of its slice from shared
//   memory and CTA 0 adds the eight partial sums:
//       key[r] = sum_v rint(2^40 * e(RN32(l_v - m))),  arg[r] = first argmax
//   The sum is an integer, so the key does not depend on the reduction order
//   and matches a scalar CPU loop bit for bit. key / 2^40 = 1 / (max softmax
//   probability) up to the rounding of e; smaller key = more confident.
// Kernel 2 (commit_select_kernel), one CTA per block: rank every masked row
//   by (key, row) and commit the first min(k, #masked): tok[r] = arg[r],
//   masked_out[r] = 0.
//
// e(x) is an fp32 exponential defined for this purpose (Cody and Waite range
// reduction, then the degree-7 Taylor polynomial of exp, all with
// round-to-nearest fused multiply-adds):
//   x < -30 -> term 0
//   t = RN(x * log2(e)), n = rint(t)
//   r = fma(-n, C1, x), r = fma(-n, C2, r)     C1 = RN32(ln 2), C2 = RN32(ln 2 - C1)
//   p = c7; p = fma(p, r, c_j), j = 6..0       c_j = RN32(1 / j!)
//   term = rint(p * 2^(n + 40))
#include <cooperative_groups.h>

#include "ptx.cuh"
#include "tt_internal.h"

namespace cg = cooperative_groups;

namespace tt {

namespace {

// RN32(1/ln 2), RN32(ln 2), RN32(ln 2 - RN32(ln 2)), RN32(1/j!)
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e430p-1f;
constexpr float kLn2Lo = -0x1.05c610p-29f;
constexpr float kInvFact2 = 0x1.000000p-1f;
constexpr float kInvFact3 = 0x1.555556p-3f;
constexpr float kInvFact4 = 0x1.555556p-5f;
constexpr float kInvFact5 = 0x1.111112p-7f;
constexpr float kInvFact6 = 0x1.6c16c2p-10f;
constexpr float kInvFact7 = 0x1.a01a02p-13f;

// Fixed-point term rint(2^40 * e(x)) for x <= 0; explicit round-to-nearest
// intrinsics so that no multiply-add is contracted differently.
__device__ __forceinline__ unsigned long long fixed_term(float x) {
    const float xc = fmaxf(x, -31.0f);
    const float n = rintf(__fmul_rn(xc, kLog2e));
    float r = __fmaf_rn(-n, kLn2Hi, xc);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = kInvFact7;
    p = __fmaf_rn(p, r, kInvFact6);
    p = __fmaf_rn(p, r, kInvFact5);
    p = __fmaf_rn(p, r, kInvFact4);
    p = __fmaf_rn(p, r, kInvFact3);
    p = __fmaf_rn(p, r, kInvFact2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const float scale = __int_as_float((static_cast<int>(n) + 40 + 127) << 23);  // 2^(n+40)
    const unsigned long long q = __float2ull_rn(__fmul_rn(p, scale));
    return x < -30.0f ? 0ull : q;
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

__global__ void __cluster_dims__(kCommitCluster, 1, 1) __launch_bounds__(kCommitThreads)
    commit_rows_kernel(const CommitParams p) {
    extern __shared__ __align__(128) float slice[];
    __shared__ __align__(8) uint64_t bars[kPieces];
    __shared__ ArgMax red_am[kCommitThreads / 32];
    __shared__ unsigned long long red_s[kCommitThreads / 32];
    __shared__ ArgMax cta_am;               // this CTA's (max, argmax), read by the cluster
    __shared__ unsigned long long cta_sum;  // this CTA's partial key, read by rank 0
    __shared__ ArgMax row_am;

    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kCommitCluster;
    const unsigned rank = cluster.block_rank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (!p.masked[row]) return;  // uniform over the cluster: all its CTAs read the same flag

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

    // Pass 1: max and first argmax of the slice, piece by piece as it lands.
    ArgMax am{-INFINITY, 0x7fffffff};
    bool ok = true;
    for (int i = 0; i < kPieces; ++i) {
        const int lo = i * per, hi = min(cnt, lo + per);
        if (hi <= lo) break;
        if (!mbar_wait(&bars[i], 0, p.timeout_ns)) { ok = false; break; }
        for (int e = lo + tid * 4; e < hi; e += kCommitThreads * 4) {
            const float4 x = *reinterpret_cast<const float4*>(slice + e);
            if (x.x > am.v) { am.v = x.x; am.i = v0 + e; }
            if (x.y > am.v) { am.v = x.y; am.i = v0 + e + 1; }
            if (x.z > am.v) { am.v = x.z; am.i = v0 + e + 2; }
            if (x.w > am.v) { am.v = x.w; am.i = v0 + e + 3; }
        }
    }
    if (!ok) {
        if (tid == 0) atomicOr(p.status, kDevWaitTimeout);
        // Let every copy already issued land before this CTA can exit.
        for (int i = 0; i < kPieces; ++i)
            if (min(cnt, i * per + per) > i * per) mbar_wait(&bars[i], 0, p.timeout_ns);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax other{__shfl_xor_sync(0xffffffffu, am.v, o), __shfl_xor_sync(0xffffffffu, am.i, o)};
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
        for (int r = 0; r < kCommitCluster; ++r) a = better(a, *cluster.map_shared_rank(&cta_am, r));
        row_am = a;
    }
    __syncthreads();
    const float m = row_am.v;

    // Pass 2: fixed-point confidence terms of the slice.
    unsigned long long acc = 0;
    if (ok) {
        for (int e = tid * 4; e < cnt; e += kCommitThreads * 4) {
            const float4 x = *reinterpret_cast<const float4*>(slice + e);
            acc += fixed_term(__fsub_rn(x.x, m));
            acc += fixed_term(__fsub_rn(x.y, m));
            acc += fixed_term(__fsub_rn(x.z, m));
            acc += fixed_term(__fsub_rn(x.w, m));
        }
    }
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

// One CTA per block: rank the still-masked rows by (key, row) and commit the
// first k of them.
__global__ void __launch_bounds__(1024) commit_select_kernel(const CommitParams p) {
    extern __shared__ __align__(8) unsigned char sel_smem[];
    unsigned long long* s_key = reinterpret_cast<unsigned long long*>(sel_smem);
    uint8_t* s_m = sel_smem + static_cast<size_t>(p.L) * 8;
    const int b = blockIdx.x;
    const size_t base = static_cast<size_t>(b) * p.L;
    for (int i = threadIdx.x; i < p.L; i += blockDim.x) {
        const uint8_t mk = p.masked[base + i];
        s_m[i] = mk;
        s_key[i] = mk ? p.key[base + i] : 0ull;
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
            p.tok[base + i] = p.arg[base + i];
            p.masked_out[base + i] = 0;
        } else {
            p.masked_out[base + i] = 1;
        }
    }
}

}  // namespace

cudaError_t launch_commit(const CommitParams& p, cudaStream_t s) {
    const size_t rows_smem = static_cast<size_t>(p.slice) * 4;
    commit_rows_kernel<<<static_cast<unsigned>(p.B * p.L) * kCommitCluster, kCommitThreads,
                         rows_smem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int threads = p.L >= 1024 ? 1024 : ((p.L + 31) / 32) * 32;
    commit_select_kernel<<<p.B, threads, static_cast<size_t>(p.L) * 9, s>>>(p);
    return cudaGetLastError();
}

cudaError_t configure_commit_kernels() {
    return cudaFuncSetAttribute(commit_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCommitSliceMax * 4);
}

}  // namespace tt
