// Per-block top-k selection of the unmask/commit step ("Nemotron-Labs-TwoTower",
// Section 2.2, Algorithm 2, confidence unmasking), shared by the commit
// kernels: once every masked row of block b has its canonical key and
// prediction, the block's masked rows are ranked by (key, row) ascending and
// the first ones commit (tok[r] = arg[r], masked_out[r] = 0; the other masked
// rows get masked_out[r] = 1). P is a parameter struct with the fields masked,
// key, arg, tok, masked_out, L, k, steps_left and kthr (see CommitParams).
#pragma once

#include "tt_internal.h"

namespace tt {
namespace sel {

constexpr int kSelChunk = 2048;  // keys staged per selection pass (shared memory)

// Commits the k most confident masked rows of block b: tok[r] = arg[r],
// masked_out[r] = 0; the block's other masked rows get masked_out[r] = 1
// (unmasked rows are written by the row's owner). Order: (key, row)
// ascending. Every masked row of the block has written its key and
// prediction (the block's last ticket was taken); reads go through L2. Run by
// one warp. All masked flags are read before any write, since masked_out may
// alias masked. n = number of masked rows in the block.
//   n <= k: every masked row commits, no ranking;
//   L <= kSelChunk: k rounds of a warp argmin over the keys staged in shared
//       memory, each round taking the smallest (key, row) above the last;
//   larger L: each row's rank is counted over the keys, chunk by chunk.
// Rows block b commits, given its n masked rows and, in threshold mode, the
// number of them whose key is <= kthr (cthr, the rows whose confidence is
// above gamma: they are the first cthr rows of the (key, row) order).
template <class P>
__device__ __forceinline__ int block_budget(const P& p, int n, int cthr) {
    if (p.steps_left <= 0) return p.k;
    return max(cthr, (n + p.steps_left - 1) / p.steps_left);
}

// L <= 256: every lane holds up to 8 rows (row 32 q + lane) in registers;
// flags, keys and predictions come in one round trip of loads.
constexpr int kSelRegRows = 8;

template <class P>
__device__ void select_block_small(const P& p, int b, int n, int lane) {
    const size_t base = static_cast<size_t>(b) * p.L;
    bool mi[kSelRegRows];
    unsigned long long ki[kSelRegRows];
    int ai[kSelRegRows];
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q) {
        const int i = q * 32 + lane;
        mi[q] = false;
        ki[q] = ~0ull;
        ai[q] = 0;
        if (i < p.L) {
            mi[q] = __ldcg(p.masked + base + i) != 0;
            ki[q] = __ldcg(p.key + base + i);
            ai[q] = __ldcg(p.arg + base + i);
        }
    }
    int cthr = 0;
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q) {
        if (!mi[q]) ki[q] = ~0ull;  // unmasked rows never rank
        cthr += (mi[q] && ki[q] <= p.kthr) ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cthr += __shfl_xor_sync(0xffffffffu, cthr, o);
    const int kb = block_budget(p, n, cthr);
    uint32_t commit = 0;  // bit q: row 32 q + lane is committed
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q)
        if (n <= kb && mi[q]) commit |= 1u << q;
    if (n > kb) {
        unsigned long long lk = 0;  // last chosen (key, row); row -1: none yet
        int lr = -1;
        for (int round = 0; round < kb; ++round) {
            unsigned long long bk = ~0ull;
            int br = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < kSelRegRows; ++q) {
                const int j = q * 32 + lane;
                const bool above = ki[q] > lk || (ki[q] == lk && j > lr);
                const bool below = ki[q] < bk || (ki[q] == bk && j < br);
                if (ki[q] != ~0ull && above && below) { bk = ki[q]; br = j; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long ok_ = __shfl_xor_sync(0xffffffffu, bk, o);
                const int orow = __shfl_xor_sync(0xffffffffu, br, o);
                if (ok_ < bk || (ok_ == bk && orow < br)) { bk = ok_; br = orow; }
            }
            if (br == 0x7fffffff) break;
            if ((br & 31) == lane) commit |= 1u << (br >> 5);
            lk = bk;
            lr = br;
        }
    }
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q) {
        const int i = q * 32 + lane;
        if (mi[q]) {
            const bool c = (commit >> q) & 1u;
            if (c) p.tok[base + i] = ai[q];
            p.masked_out[base + i] = c ? 0 : 1;
        }
    }
}

template <class P>
__device__ void select_block(const P& p, int b, int n, unsigned long long* s_key,
                             uint32_t* s_mbits, uint32_t* s_cbits, int lane) {
    const size_t base = static_cast<size_t>(b) * p.L;
    const int nw = (p.L + 31) / 32;
    int cthr = 0;
    for (int w = 0; w < nw; ++w) {
        const int i = w * 32 + lane;
        const bool mi = i < p.L && __ldcg(p.masked + base + i) != 0;
        cthr += (mi && p.steps_left > 0 && __ldcg(p.key + base + i) <= p.kthr) ? 1 : 0;
        const uint32_t mb = __ballot_sync(0xffffffffu, mi);
        if (lane == 0) s_mbits[w] = mb;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cthr += __shfl_xor_sync(0xffffffffu, cthr, o);
    const int kb = block_budget(p, n, cthr);
    if (lane == 0)
        for (int w = 0; w < nw; ++w) s_cbits[w] = n <= kb ? s_mbits[w] : 0u;
    __syncwarp();
    if (n > kb && p.L <= kSelChunk) {
        for (int j = lane; j < p.L; j += 32)
            s_key[j] = (s_mbits[j >> 5] >> (j & 31)) & 1u ? __ldcg(p.key + base + j) : ~0ull;
        __syncwarp();
        unsigned long long lk = 0;  // last chosen (key, row); row -1: none yet
        int lr = -1;
        for (int round = 0; round < kb; ++round) {
            unsigned long long bk = ~0ull;
            int br = 0x7fffffff;
            for (int j = lane; j < p.L; j += 32) {
                const unsigned long long kj = s_key[j];
                const bool above = kj > lk || (kj == lk && j > lr);
                const bool below = kj < bk || (kj == bk && j < br);
                if (kj != ~0ull && above && below) { bk = kj; br = j; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long ok_ = __shfl_xor_sync(0xffffffffu, bk, o);
                const int orow = __shfl_xor_sync(0xffffffffu, br, o);
                if (ok_ < bk || (ok_ == bk && orow < br)) { bk = ok_; br = orow; }
            }
            if (br == 0x7fffffff) break;
            if (lane == 0) s_cbits[br >> 5] |= 1u << (br & 31);
            lk = bk;
            lr = br;
        }
    } else if (n > kb) {
        for (int w = 0; w < nw; ++w) {
            const int i = w * 32 + lane;
            const bool mi = (s_mbits[w] >> lane) & 1u;
            const unsigned long long ki = mi ? __ldcg(p.key + base + i) : 0ull;
            int rank = 0;
            for (int j0 = 0; j0 < p.L; j0 += kSelChunk) {
                const int cn = min(kSelChunk, p.L - j0);
                __syncwarp();
                for (int j = lane; j < cn; j += 32)
                    s_key[j] = (s_mbits[(j0 + j) >> 5] >> ((j0 + j) & 31)) & 1u
                                   ? __ldcg(p.key + base + j0 + j)
                                   : ~0ull;
                __syncwarp();
                const int lim = i - j0;  // rows j0 + j < i win ties
                for (int j = 0; j < cn; ++j) {
                    const unsigned long long kj = s_key[j];
                    rank += (kj < ki || (kj == ki && j < lim)) ? 1 : 0;
                }
            }
            const uint32_t cb = __ballot_sync(0xffffffffu, mi && rank < kb);
            if (lane == 0) s_cbits[w] = cb;
        }
    }
    __syncwarp();
    for (int w = 0; w < nw; ++w) {
        const int i = w * 32 + lane;
        if ((s_mbits[w] >> lane) & 1u) {
            const bool c = (s_cbits[w] >> lane) & 1u;
            if (c) p.tok[base + i] = __ldcg(p.arg + base + i);
            p.masked_out[base + i] = c ? 0 : 1;
        }
    }
    __syncwarp();
}


}  // namespace sel
}  // namespace tt
