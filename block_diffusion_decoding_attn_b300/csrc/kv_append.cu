// Context-tower cache update after a block is committed ("Nemotron-Labs-TwoTower",
// Section 2.1, Algorithm 1, the context update after a commit): the committed block's keys
// and values of this layer join the prefix cache behind the positions already
// there, and the cache length grows by L.
//
// A plain HBM copy: k_blk/v_blk [B][L][Hkv][D] -> k_ctx/v_ctx [B][Hkv][cap][D]
// at rows ctx_len[b] .. ctx_len[b] + L - 1. Each thread moves 16-byte pieces;
// for a fixed (l, kv head) the D/8 pieces of a row are contiguous on both sides.
// The length update is a second launch, so that no copy can read a length
// already advanced.
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kAppendPer = 4;  // 16-byte pieces per thread

// A block that does not fit (ctx_len[b] outside [0, cap - L]) is not copied
// and its length is not advanced; the call's status gets kDevCtxLenRange.
__device__ __forceinline__ bool fits(int C, int L, int cap) { return C >= 0 && C <= cap - L; }

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const KvAppendParams p) {
    const int b = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const int C = p.ctx_len[b];
    if (!fits(C, p.L, p.ctx_cap)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && !is_v) atomicOr(p.status, kDevCtxLenRange);
        return;
    }
    const int per_row = p.D / 8;  // 16-byte pieces per (l, kv head) row
    const long n = static_cast<long>(p.L) * p.Hkv * per_row;
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? p.v_blk : p.k_blk) +
                       static_cast<size_t>(b) * n;
    uint4* dst = reinterpret_cast<uint4*>(is_v ? p.v_ctx : p.k_ctx);
    const long first = (static_cast<long>(blockIdx.x) * kAppendThreads) * kAppendPer + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kAppendPer; ++u) {
        const long i = first + static_cast<long>(u) * kAppendThreads;
        if (i >= n) break;
        const int piece = static_cast<int>(i % per_row);
        const long rowi = i / per_row;  // l * Hkv + kv head
        const int kvh = static_cast<int>(rowi % p.Hkv);
        const int l = static_cast<int>(rowi / p.Hkv);
        const size_t d = ((static_cast<size_t>(b) * p.Hkv + kvh) * p.ctx_cap + C + l) * per_row + piece;
        dst[d] = __ldcs(src + i);
    }
}

__global__ void __launch_bounds__(256) ctx_len_advance_kernel(const KvAppendParams p) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int C = p.ctx_len[b];
    if (fits(C, p.L, p.ctx_cap)) p.ctx_len[b] = C + p.L;
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendParams& p, cudaStream_t s) {
    if (p.B == 0) return cudaSuccess;
    const long n = static_cast<long>(p.L) * p.Hkv * (p.D / 8);
    const long per_block = static_cast<long>(kAppendThreads) * kAppendPer;
    const dim3 grid(static_cast<unsigned>((n + per_block - 1) / per_block), static_cast<unsigned>(p.B), 2);
    kv_append_kernel<<<grid, kAppendThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ctx_len_advance_kernel<<<(p.B + 255) / 256, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tt
