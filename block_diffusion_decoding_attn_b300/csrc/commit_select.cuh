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
//   L <= 256 (select_block_small): rounds of a warp minimum over per-lane
//       sorted lists (binary search on the key for large budgets);
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

// L <= 256 (select_block_small): lane l holds rows 8 l .. 8 l + 7 in
// registers (flags, keys and predictions in one round trip of loads). Up to
// kSelRounds commits: each lane sorts its 8 (key, row) pairs, then every round
// takes the warp minimum of the lanes' heads with three redux.sync minima
// (key high word, key low word, lane: rows are lane-major, so the lowest lane
// holds the lowest row among equal keys) and the winning lane pops its head.
// More commits: a binary search for the kb-th smallest key with ballots, then
// the tied rows at that key in row order.
constexpr int kSelRegRows = 8;
constexpr int kSelRounds = 96;

__device__ __forceinline__ bool key_row_less(unsigned long long ka, int ra, unsigned long long kb,
                                             int rb) {
    return ka < kb || (ka == kb && ra < rb);
}

template <class P>
__device__ void select_block_small(const P& p, int b, int n, int lane) {
    const size_t base = static_cast<size_t>(b) * p.L;
    unsigned long long key[kSelRegRows];
    int arg[kSelRegRows];
    uint32_t mbits = 0;  // bit q: row 8 lane + q is masked
    {
        uint8_t m[kSelRegRows];
        unsigned long long k[kSelRegRows];
#pragma unroll
        for (int q = 0; q < kSelRegRows; ++q) {
            const int i = min(lane * kSelRegRows + q, p.L - 1);
            m[q] = __ldcg(p.masked + base + i);
            k[q] = __ldcg(p.key + base + i);
            arg[q] = __ldcg(p.arg + base + i);
        }
#pragma unroll
        for (int q = 0; q < kSelRegRows; ++q) {
            const bool ok = lane * kSelRegRows + q < p.L && m[q] != 0;
            mbits |= ok ? (1u << q) : 0u;
            key[q] = ok ? k[q] : ~0ull;  // a masked row's key is below 2^63
        }
    }
    int cthr = 0;
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q) cthr += key[q] <= p.kthr ? 1 : 0;
    cthr = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cthr)));
    const int kb = block_budget(p, n, cthr);
    uint32_t cbits = mbits;  // bit q: row 8 lane + q commits
    if (n > kb && kb <= kSelRounds) {
        unsigned long long sk[kSelRegRows];
        int sq[kSelRegRows];
#pragma unroll
        for (int q = 0; q < kSelRegRows; ++q) {
            sk[q] = key[q];
            sq[q] = q;
        }
        // odd-even transposition sort of the lane's pairs
#pragma unroll
        for (int pass = 0; pass < kSelRegRows; ++pass) {
#pragma unroll
            for (int q = pass & 1; q + 1 < kSelRegRows; q += 2) {
                if (key_row_less(sk[q + 1], sq[q + 1], sk[q], sq[q])) {
                    const unsigned long long tk = sk[q];
                    sk[q] = sk[q + 1];
                    sk[q + 1] = tk;
                    const int tq = sq[q];
                    sq[q] = sq[q + 1];
                    sq[q + 1] = tq;
                }
            }
        }
        cbits = 0;
        for (int round = 0; round < kb; ++round) {
            const unsigned hi = static_cast<unsigned>(sk[0] >> 32), lo = static_cast<unsigned>(sk[0]);
            const unsigned m1 = __reduce_min_sync(0xffffffffu, hi);
            const unsigned m2 = __reduce_min_sync(0xffffffffu, hi == m1 ? lo : 0xffffffffu);
            const unsigned me = (hi == m1 && lo == m2) ? static_cast<unsigned>(lane) : 0xffffffffu;
            if (static_cast<unsigned>(lane) == __reduce_min_sync(0xffffffffu, me)) {
                cbits |= 1u << sq[0];
#pragma unroll
                for (int q = 0; q + 1 < kSelRegRows; ++q) {
                    sk[q] = sk[q + 1];
                    sq[q] = sq[q + 1];
                }
                sk[kSelRegRows - 1] = ~0ull;
            }
        }
    } else if (n > kb) {
        // smallest T with #(key <= T) >= kb; unselected rows (key ~0) never count
        unsigned long long lo = 0, hi = ~0ull - 1;
        while (lo < hi) {
            const unsigned long long mid = lo + ((hi - lo) >> 1);
            int c = 0;
#pragma unroll
            for (int q = 0; q < kSelRegRows; ++q) c += __popc(__ballot_sync(0xffffffffu, key[q] <= mid));
            if (c >= kb) hi = mid;
            else lo = mid + 1;
        }
        int clt = 0, before = 0;  // rows below T; rows at T in lower lanes
        const uint32_t lower_lanes = (1u << lane) - 1u;
#pragma unroll
        for (int q = 0; q < kSelRegRows; ++q) {
            clt += __popc(__ballot_sync(0xffffffffu, key[q] < lo));
            before += __popc(__ballot_sync(0xffffffffu, key[q] == lo) & lower_lanes);
        }
        cbits = 0;
#pragma unroll
        for (int q = 0; q < kSelRegRows; ++q) {
            const bool tie = key[q] == lo;
            if (key[q] < lo || (tie && clt + before < kb)) cbits |= 1u << q;
            before += tie ? 1 : 0;
        }
    }
#pragma unroll
    for (int q = 0; q < kSelRegRows; ++q) {
        if ((mbits >> q) & 1u) {
            const size_t i = base + lane * kSelRegRows + q;
            const bool c = (cbits >> q) & 1u;
            if (c) p.tok[i] = arg[q];
            p.masked_out[i] = c ? 0 : 1;
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
