// Unmask/commit step of the TwoTower sampler ("Nemotron-Labs-TwoTower",
// Section 2.2, Algorithm 2, confidence unmasking) with a fixed budget of k
// commits per block per step. One launch.
//
// For every still-masked row r:
//     m = max_v l_v,  arg[r] = lowest v with l_v == m (greedy prediction)
//     key[r] = sum_v rint(2^40 * e(RN32(l_v - m)))
// The key is an integer, so it does not depend on the reduction order and
// matches a scalar CPU loop bit for bit; key / 2^40 = 1 / (max softmax
// probability) up to the rounding of e, so a smaller key is more confident.
// When every row of a block is done, the block's masked rows are ranked by
// (key, row) and the first min(k, #masked) are committed: tok[r] = arg[r],
// masked_out[r] = 0.
//
// Layout of the work: a persistent grid of 4-CTA clusters. Cluster c owns a
// contiguous share of the masked rows (by ordinal; the shares differ by at
// most one row); CTA j of the cluster owns the j-th quarter of each of its
// rows (128 KB at V = 131072). Per CTA (16 warps):
//   producer (warp 12): for each owned masked row, bulk TMA copies of the
//       CTA's quarter in 64 KB chunks into a 3-slot shared-memory ring (L2
//       evict-first); unmasked rows are only marked in masked_out;
//   pass 1 (warps 0-3, one per TMEM lane quarter): streams each row's chunks
//       from shared memory into one of two TMEM row slots (128 lanes x 256
//       columns = one quarter row), keeping the slice max / first argmax /
//       min, and frees each ring slot at once;
//   slice sender (warp 14): sends the CTA's slice result to all 4 CTAs as a
//       one-way st.async message on their exchange mbarrier;
//   pass 2 (warps 4-11): once the 4 slice results of the row are in (row max
//       m, prediction), reads the slot back 32 columns at a time and sums the
//       fixed-point terms, then frees the slot;
//   key sender (warp 15): sends the CTA's partial key to CTA 0 the same way;
//   collector (warp 13 of CTA 0): adds each row's 4 partial keys, writes
//       key/arg; per block it takes one ticket for all of the cluster's rows
//       of the block (the count is the block's number of masked rows); the
//       warp that completes the count ranks the block's masked rows and
//       commits.
// Pass 1 and the exchange of row i + 1 run while pass 2 works on row i.

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
#include <atomic>

#include "ptx.cuh"
#include "tt_internal.h"

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
constexpr unsigned kMagic23Bits = 0x4B400000u;
constexpr unsigned kMagic43Bits = 0x55400000u;

constexpr int kSlots = 3;                 // ring depth: 64 KB chunks landing per CTA
constexpr int kChunk = 16384;             // logits per ring slot
constexpr int kSliceMax = 2 * kChunk;               // 32768 logits per CTA
constexpr int kRowCols = kSliceMax / 128;           // 256 TMEM columns per row slot, 2 slots
constexpr int kP1Warps = 4;               // pass 1: warps 0-3 (one per TMEM lane quarter)
constexpr int kP2Warps = 8;               // pass 2: warps 4-11
constexpr int kP1Threads = kP1Warps * 32;
constexpr int kProducerWarp = kP1Warps + kP2Warps;  // warp 12
constexpr int kCollectorWarp = kProducerWarp + 1;   // warp 13 (CTA 0 only)
constexpr int kAmSenderWarp = kCollectorWarp + 1;   // warp 14: slice results -> the cluster
constexpr int kSumSenderWarp = kAmSenderWarp + 1;   // warp 15: partial keys -> CTA 0
constexpr int kP1PerChunk = kChunk / kP1Threads;    // logits per pass-1 thread per chunk
constexpr int kP2Cols = kRowCols / (kP2Warps / 4);  // TMEM columns per pass-2 thread
constexpr int kThreads = (kSumSenderWarp + 1) * 32;
constexpr int kXchg = 8;                  // exchange slots (rows in flight in the cluster)
constexpr int kSelChunk = 2048;           // keys staged per selection pass
static_assert(kSliceMax == kCommitSliceMax, "slice per CTA");
static_assert(2 * kRowCols == 512, "two row slots fill the TMEM");

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
__device__ __forceinline__ f2 ffma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 fadd2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 fsub2(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Adds the fixed-point terms of x0, x1 (RN32(l - m) clamped below at -31;
// terms below -28.4 round to 0 either way) to the accumulators:
//   sum of terms = (hi - cnt * kMagic43Bits) * 2^20 + (lo - cnt * kMagic23Bits)
// (mod 2^32 each), with cnt the number of terms added; the constant offsets
// are taken out once at the end.
__device__ __forceinline__ void add_terms(f2 x, unsigned& hi, unsigned& lo) {
    const f2 nb = ffma2(x, dup(kLog2e), dup(kMagic23));  // 1.5*2^23 + n
    const f2 n = fsub2(nb, dup(kMagic23));
    f2 r = ffma2(n, dup(-kLn2Hi), x);
    r = ffma2(n, dup(-kLn2Lo), r);
    f2 p = ffma2(dup(kC7), r, dup(kC6));
    p = ffma2(p, r, dup(kC5));
    p = ffma2(p, r, dup(kC4));
    p = ffma2(p, r, dup(kC3));
    p = ffma2(p, r, dup(kC2));
    p = ffma2(p, r, dup(kC0));
    p = ffma2(p, r, dup(kC0));  // 2^40 * p(r), in [2^39.5, 2^40.5]
    float p0, p1, nb0, nb1;
    upk(p, p0, p1);
    upk(nb, nb0, nb1);
    // y = p * 2^n: add n to the exponent field; (bits(nb) << 23) == (n << 23) mod 2^32.
    const f2 y = pk(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(nb0) << 23)),
                    __uint_as_float(__float_as_uint(p1) + (__float_as_uint(nb1) << 23)));
    const f2 a = fadd2(y, dup(kMagic43));               // 1.5*2^43 + 2^20 * round(y / 2^20)
    const f2 rem = fsub2(y, fsub2(a, dup(kMagic43)));   // exact, |rem| <= 2^19
    const f2 b = fadd2(rem, dup(kMagic23));             // 1.5*2^23 + rint(rem)
    float a0, a1, b0, b1;
    upk(a, a0, a1);
    upk(b, b0, b1);
    hi += __float_as_uint(a0) + __float_as_uint(a1);
    lo += __float_as_uint(b0) + __float_as_uint(b1);
}

// (value, index) as one orderable 64-bit word: a larger value wins, equal
// values go to the lower index. -0.0 is folded into +0.0 first (they compare
// equal). 0 is below every encoded pair.
__device__ __forceinline__ unsigned long long enc_argmax(float v, int i) {
    unsigned u = __float_as_uint(v + 0.0f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<unsigned>(i));
}
__device__ __forceinline__ float dec_value(unsigned long long e) {
    unsigned u = static_cast<unsigned>(e >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ int dec_index(unsigned long long e) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<unsigned>(e));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One group of 32 logits of a pass-1 thread: float4 u8 = 0..7 of the group at
// ring offsets e0 + 4 * kP1Threads * u8, i.e. in slice order for the thread.
// Returns the group maximum, folds the group minimum into mn and leaves the
// raw bits in rr in the same order (TMEM columns 4 u8 + j). kChecked: offsets
// at or past n (the end of the slice in this chunk) read as -inf.
template <bool kChecked>
__device__ __forceinline__ float p1_group(const float* sl, int e0, int n, float& mn,
                                          uint32_t (&rr)[32]) {
    float a0 = -INFINITY, a1 = -INFINITY, b0 = mn, b1 = INFINITY;
#pragma unroll
    for (int u8 = 0; u8 < 8; ++u8) {
        const int e = e0 + 4 * kP1Threads * u8;
        float4 x;
        if (kChecked && e >= n) x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        else x = *reinterpret_cast<const float4*>(sl + e);
        a0 = max3(a0, x.x, x.y);
        a1 = max3(a1, x.z, x.w);
        b0 = min3(b0, x.x, x.y);
        b1 = min3(b1, x.z, x.w);
        rr[4 * u8 + 0] = __float_as_uint(x.x);
        rr[4 * u8 + 1] = __float_as_uint(x.y);
        rr[4 * u8 + 2] = __float_as_uint(x.z);
        rr[4 * u8 + 3] = __float_as_uint(x.w);
    }
    mn = fminf(b0, b1);
    return fmaxf(a0, a1);
}

__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int o) {
    return __shfl_xor_sync(0xffffffffu, v, o);
}

// One exchange message: two 64-bit words, written by st.async (16 bytes).
struct alignas(16) XchgIn {
    unsigned long long a, b;
};
constexpr uint32_t kXchgBytes = kCommitCluster * sizeof(XchgIn);  // per row and barrier

struct CommitShared {
    uint64_t full[kSlots];      // producer -> pass 1: chunk landed
    uint64_t empty[kSlots];     // pass 1 -> producer: slot free (one arrival per pass-1 warp)
    uint64_t tfree[2];          // pass 2 -> pass 1: TMEM row slot free (one arrival per pass-2 warp)
    uint64_t p1_done[kXchg];    // pass 1 -> slice sender: the row's per-warp results are written
    uint64_t p2_done[kXchg];    // pass 2 -> key sender: the row's per-warp partial keys are written
    uint64_t am_bar[kXchg];     // 16 bytes from each CTA: its slice (argmax code, min)
    uint64_t sum_bar[kXchg];    // 16 bytes from each CTA at CTA 0: (partial key, prediction)
    uint64_t col_done[kXchg];   // CTA 0: the collector has finished the row
    XchgIn am_in[kXchg][kCommitCluster];   // (argmax code, slice min) from the cluster's CTAs
    XchgIn sum_in[kXchg][kCommitCluster];  // (partial key, prediction) (CTA 0 only)
    int row_arg[kXchg];                                 // pass 2 -> key sender: prediction
    unsigned long long red_am[kXchg][kP1Warps];
    float red_min[kXchg][kP1Warps];
    unsigned long long red_sum[kXchg][kP2Warps];
    int xchg_err;           // a receiver gave up waiting for an exchange
    int total;              // masked rows of this cluster
    int row0;               // first row of this cluster's range
    int wsum[kThreads / 32];  // start-up scan: masked rows per warp
    uint32_t tmem;          // TMEM base address (512 columns)
};

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
__device__ __forceinline__ int block_budget(const CommitParams& p, int n, int cthr) {
    if (p.steps_left <= 0) return p.k;
    return max(cthr, (n + p.steps_left - 1) / p.steps_left);
}

// L <= 256: every lane holds up to 8 rows (row 32 q + lane) in registers;
// flags, keys and predictions come in one round trip of loads.
constexpr int kSelRegRows = 8;

__device__ void select_block_small(const CommitParams& p, int b, int n, int lane) {
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

__device__ void select_block(const CommitParams& p, int b, int n, unsigned long long* s_key,
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

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* a, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned* a, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Counters of one call (zero between calls).
constexpr int kCtrStarted = 0;   // clusters past their start-up mask scan
constexpr int kCtrFinished = 1;  // clusters done
constexpr int kCtrTickets = 2;   // block b's ticket at kCtrTickets + b

// Masked rows of block b (read by one warp).
__device__ int count_masked(const CommitParams& p, int b, int lane) {
    const uint8_t* m = p.masked + static_cast<size_t>(b) * p.L;
    int c = 0;
    for (int i = lane; i < p.L; i += 32) c += __ldcg(m + i) != 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
}

__global__ void __cluster_dims__(kCommitCluster, 1, 1) __launch_bounds__(kThreads, 1)
    commit_kernel(const CommitParams p) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ CommitShared sh;
    float* ring = reinterpret_cast<float*>(dyn);
    unsigned char* sel_base = dyn + static_cast<size_t>(kSlots) * kChunk * 4;
    unsigned long long* s_key = reinterpret_cast<unsigned long long*>(sel_base);
    uint32_t* s_mbits = reinterpret_cast<uint32_t*>(sel_base + kSelChunk * 8);
    uint32_t* s_cbits = s_mbits + kCommitMaxL / 32;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());
    const int rows = p.B * p.L;
    const int v0 = static_cast<int>(rank) * p.slice;
    const int cnt = max(0, min(p.slice, p.V - v0));  // this CTA's logits per row (multiple of 4)
    const int nchunks = (cnt + kChunk - 1) / kChunk;  // ring entries per row (0 if cnt == 0)
    const uint64_t limit = p.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kP1Warps);
        }
        mbar_init(&sh.tfree[0], kP2Warps);
        mbar_init(&sh.tfree[1], kP2Warps);
        for (int q = 0; q < kXchg; ++q) {
            mbar_init(&sh.p1_done[q], kP1Warps);
            mbar_init(&sh.p2_done[q], kP2Warps);
            mbar_init(&sh.am_bar[q], 1);
            mbar_init(&sh.sum_bar[q], 1);
            mbar_init(&sh.col_done[q], 1);
        }
        fence_mbar_init();
        // Each exchange barrier expects the messages of its first row; the
        // receiver re-arms it for row + kXchg once it has read a row.
        for (int q = 0; q < kXchg; ++q) {
            mbar_arrive_expect_tx(&sh.am_bar[q], kXchgBytes);
            mbar_arrive_expect_tx(&sh.sum_bar[q], kXchgBytes);
        }
        sh.xchg_err = 0;
    }
    if (warp == 0) {
        tmem_alloc(&sh.tmem, 512);
        tmem_relinquish();
    }
    // The cluster's share of the rows: the masked rows with ordinals
    // [cid * M / ncl, (cid + 1) * M / ncl) (M = masked rows in total), and the
    // unmasked rows from the cluster's first masked row (row 0 for cluster 0)
    // up to the next cluster's first one. Every role of every CTA of the
    // cluster walks these rows in order; contiguous shares keep the blocks a
    // cluster touches (and so its block tickets) few. Thread tid counts
    // rows [tid * S, tid * S + S); a block-wide scan of the counts finds M and
    // the thread that holds ordinal cid * M / ncl finds its row.
    {
        const int S = (rows + kThreads - 1) / kThreads;
        const int r_lo = min(rows, tid * S), r_hi = min(rows, r_lo + S);
        int c = 0;
        for (int r = r_lo; r < r_hi; ++r) c += __ldcg(p.masked + r) != 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) sh.wsum[warp] = incl;
        __syncthreads();
        int wpre = 0, mtot = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            const int v = sh.wsum[w];
            wpre += w < warp ? v : 0;
            mtot += v;
        }
        const int excl = wpre + incl - c;
        const int o0 = static_cast<int>(static_cast<long long>(cid) * mtot / ncl);
        const int o1 = static_cast<int>(static_cast<long long>(cid + 1) * mtot / ncl);
        if (tid == 0) {
            sh.total = o1 - o0;
            if (cid == 0 || o0 >= mtot) sh.row0 = cid == 0 ? 0 : rows;
        }
        if (cid > 0 && o0 < mtot && excl <= o0 && o0 < excl + c) {
            int seen = excl;
            for (int r = r_lo; r < r_hi; ++r)
                if (__ldcg(p.masked + r) != 0 && seen++ == o0) {
                    sh.row0 = r;
                    break;
                }
        }
    }
    tc_fence_before();
    // Every CTA's barriers are initialised before any remote arrival.
    cluster_sync_all();
    tc_fence_after();
    // The cluster's scans are over. When masked_out is the masked buffer, no
    // block selection writes the mask before every cluster has scanned it (the
    // selecting warp waits for this count to reach the number of clusters).
    if (rank == 0 && tid == 0) red_add_release_gpu(p.counters + kCtrStarted, 1u);

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- producer
        // The masked rows of this cluster go through the ring in row order,
        // max(nchunks, 1) entries each; the unmasked ones are only marked in
        // masked_out.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const int per_row = max(nchunks, 1);
            int it = 0;  // ring entries issued
            bool ok = true;
            const int total = sh.total;
            int done = 0;
            for (int r = sh.row0; r < rows && ok; ++r) {
                // masked may alias masked_out: this read precedes the block's
                // selection, which waits for this row's ticket.
                if (__ldcg(p.masked + r) == 0) {
                    if (rank == 0) p.masked_out[r] = 0;
                    continue;
                }
                if (done == total) break;  // the next cluster's first row
                ++done;
                for (int c = 0; c < per_row; ++c, ++it) {
                    const int s = it % kSlots;
                    if (it >= kSlots && !mbar_wait(&sh.empty[s], ((it / kSlots) - 1) & 1, limit)) {
                        ok = false;
                        break;
                    }
                    const int lo = c * kChunk, n = min(kChunk, cnt - lo);
                    if (n > 0) {
                        mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(n) * 4);
                        bulk_load(ring + static_cast<size_t>(s) * kChunk,
                                  p.logits + static_cast<size_t>(r) * p.V + v0 + lo,
                                  static_cast<uint32_t>(n) * 4, &sh.full[s], pol);
                    } else {
                        mbar_arrive(&sh.full[s]);
                    }
                }
            }
            if (!ok) atomicOr(p.status, kDevWaitTimeout);
            // Let the copies already issued land before the CTA can exit (an
            // entry is issued only once the one kSlots before it was consumed, so
            // at most the last kSlots can be in flight; after a normal run they
            // have all landed). Also when a consumer gave up instead.
            const uint64_t dl = drain_limit(limit);
            for (int j = it - kSlots < 0 ? 0 : it - kSlots; j < it; ++j)
                mbar_wait(&sh.full[j % kSlots], (j / kSlots) & 1, dl);
        }
        __syncwarp();
    } else if (warp == kCollectorWarp) {
        // ---------------------------------------------------------------- collector
        // CTA 0: adds each row's partial keys and writes key / prediction.
        // The cluster's rows of one block are consecutive in its row order;
        // once they are all written, it adds their number to the block's
        // ticket counter, and the cluster that completes the count (the
        // block's number of masked rows) selects the block.
        if (rank == 0) {
            int it = 0, cb = -1, cnum = 0, cmine = 0;
            bool ok = true;
            auto flush = [&]() {
                int last = 0;
                if (lane == 0) {
                    // acq_rel: the rows' key / arg are visible before the ticket;
                    // the last ticket sees every other cluster's rows.
                    unsigned* tk = p.counters + kCtrTickets + cb;
                    const unsigned t = atom_add_acq_rel_gpu(tk, static_cast<unsigned>(cmine));
                    last = t + static_cast<unsigned>(cmine) == static_cast<unsigned>(cnum);
                    if (last) *tk = 0;  // no other ticket of this call remains
                    if (last && p.alias) {
                        // the mask is written in place: every cluster has scanned it first
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire_gpu(p.counters + kCtrStarted) < static_cast<unsigned>(ncl)) {
                            if (globaltimer_ns() - t0 > limit) {
                                last = 0;
                                ok = false;
                                break;
                            }
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();  // every lane reads the other clusters' rows after the ticket
                    if (p.L <= 32 * kSelRegRows) select_block_small(p, cb, cnum, lane);
                    else select_block(p, cb, cnum, s_key, s_mbits, s_cbits, lane);
                }
            };
            const int total = sh.total;
            for (int r = sh.row0; r < rows && it < total; ++r) {
                if (__ldcg(p.masked + r) == 0) continue;
                const int q = it % kXchg;
                if (!mbar_wait_cluster(&sh.sum_bar[q], (it / kXchg) & 1, limit)) {
                    ok = false;
                    if (lane == 0) sh.xchg_err = 1;
                    break;
                }
                unsigned long long key = 0;
#pragma unroll
                for (int j = 0; j < kCommitCluster; ++j) key += sh.sum_in[q][j].a;
                const int arg = static_cast<int>(sh.sum_in[q][0].b);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sh.sum_bar[q], kXchgBytes);  // for row it + kXchg
                    p.key[r] = key;
                    p.arg[r] = arg;
                    mbar_arrive(&sh.col_done[q]);
                }
                ++it;
                const int b = r / p.L;
                if (b != cb) {
                    if (cb >= 0) flush();
                    if (!ok) break;
                    cb = b;
                    cmine = 0;
                    cnum = count_masked(p, b, lane);
                }
                ++cmine;
            }
            if (ok && cb >= 0) flush();
            if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- pass 1 / pass 2
        // Rows of the cluster's sequence alternate between the two TMEM row
        // slots (256 columns each). Pass 1 (warps 0-3) drains a row's chunks
        // from the ring into its slot, taking the slice max / first argmax /
        // min; warp 14 sends the result to the cluster. Pass 2 (warps 4-11)
        // waits for the cluster's results of that row, sums its fixed-point
        // terms from TMEM and frees the slot; warp 15 sends the partial key to
        // CTA 0. So pass 1 of row i + 1 and the exchange run while pass 2
        // works on row i, and no computing warp waits for a DSMEM send. The
        // per-warp results of row i go through slot i % kXchg of shared
        // memory; that slot is written again only kXchg rows later, after
        // the exchange of those rows (whose CTA-0 side waits for the
        // collector to finish row i) has consumed it. Every wait is bounded;
        // a role whose wait gives up leaves its loop, and the others' waits
        // then give up in turn.
        const int per_row = max(nchunks, 1);  // ring entries per row
        const int total = sh.total;
        bool ok = true;
        if (warp < kP1Warps) {
            // ------------------------------------------------------------ pass 1
            // Thread pt writes TMEM lane pt % 128. Chunk c of the row goes to
            // columns 128 c .. 128 c + 127 of the slot, kP1PerChunk of them
            // from 128 c + kP1PerChunk * (pt / 128) for this thread, in groups
            // of 32: float4 u of the chunk (slice element c * kChunk +
            // 4 * (u * kP1Threads + pt)) in 4 columns from there + 4 u, so the
            // columns run in slice order for every thread. (Pass 2 only sums,
            // so it reads them in any order.) A thread keeps only its maximum
            // and the first group that reaches it; once the row is in, the
            // warp reads those groups back from TMEM (once per distinct group
            // among the lanes holding the warp maximum) to find the first
            // element equal to it.
            const int pt = tid;
            const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
            const int csub = kP1PerChunk * (pt / 128);
            for (int seq = 0; seq < total && ok; ++seq) {
                const int t = seq & 1;
                const int q = seq % kXchg;
                if (seq >= 2) ok = mbar_wait(&sh.tfree[t], ((seq >> 1) - 1) & 1, limit);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tb = sh.tmem + lane_off + static_cast<uint32_t>(t * kRowCols + csub);
                float best = -INFINITY, mn = INFINITY;
                int bcol = -1;  // column (from tb) of the group with the thread's first maximum
                int it = seq * per_row;
                for (int c = 0; c < per_row && ok; ++c, ++it) {
                    const int s = it % kSlots;
                    ok = __all_sync(0xffffffffu, mbar_wait(&sh.full[s], (it / kSlots) & 1, limit));
                    if (!ok) break;
                    const float* sl = ring + static_cast<size_t>(s) * kChunk;
                    const int n = cnt - c * kChunk;  // logits of this chunk (may exceed kChunk)
                    const bool whole = n >= kChunk;
#pragma unroll 1
                    for (int h = 0; h < kP1PerChunk / 32; ++h) {  // groups of 32 logits
                        uint32_t rr[32];
                        const int e0 = 4 * (8 * h * kP1Threads + pt);
                        const float hb = whole ? p1_group<false>(sl, e0, n, mn, rr)
                                               : p1_group<true>(sl, e0, n, mn, rr);
                        if (hb > best) {
                            best = hb;
                            bcol = 128 * c + 32 * h;
                        }
                        tmem_st32(tb + 128 * c + 32 * h, rr);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.empty[s]);  // this warp is done with the slot
                }
                if (!ok) break;
                float wmax = best;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                }
                // No lane has a group if the warp's logits are all -inf (or NaN):
                // then the warp offers no candidate (0).
                unsigned long long am = 0ull;
                unsigned cand = __ballot_sync(0xffffffffu, bcol >= 0 && best == wmax);
                while (cand != 0u) {
                    const int g = __shfl_sync(0xffffffffu, bcol, __ffs(cand) - 1);
                    uint32_t rr[32];
                    tmem_ld32(tb + g, rr);  // this thread's own stores (waited on)
                    if (((cand >> lane) & 1u) && bcol == g) {
                        int k = 31;
#pragma unroll
                        for (int j = 30; j >= 0; --j)
                            if (__uint_as_float(rr[j]) == wmax) k = j;
                        const int e = (g / 128) * kChunk +
                                      4 * ((8 * ((g % 128) / 32) + k / 4) * kP1Threads + pt) + (k & 3);
                        am = enc_argmax(wmax, v0 + e);
                    }
                    cand &= ~__ballot_sync(0xffffffffu, bcol == g);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) am = max(am, shfl_xor64(am, o));
                tc_fence_before();  // the row's TMEM stores (waited on) before the arrival
                __syncwarp();
                if (lane == 0) {
                    sh.red_am[q][warp] = am;
                    sh.red_min[q][warp] = mn;
                    mbar_arrive(&sh.p1_done[q]);
                }
            }
        } else if (warp < kP1Warps + kP2Warps) {
            // ------------------------------------------------------------ pass 2
            // Warp pw reads TMEM lanes 32 (pw % 4) .. + 31 and kP2Cols columns
            // of the slot from kP2Cols * (pw / 4) (inside chunk
            // kP2Cols * (pw / 4) / 128 of the row).
            const int pw = warp - kP1Warps;
            const int c0w = kP2Cols * (pw / 4);
            const uint32_t lane_off = static_cast<uint32_t>((warp % 4) * 32) << 16;
            const int ncol = c0w / 128 < nchunks ? kP2Cols : 0;
            for (int seq = 0; seq < total && ok; ++seq) {
                const int t = seq & 1;
                const int q = seq % kXchg;
                ok = __all_sync(0xffffffffu, mbar_wait_cluster(&sh.am_bar[q], (seq / kXchg) & 1, limit));
                if (!ok) {
                    if (lane == 0) sh.xchg_err = 1;
                    break;
                }
                tc_fence_after();
                unsigned long long rm = sh.am_in[q][0].a;
#pragma unroll
                for (int k = 1; k < kCommitCluster; ++k) rm = max(rm, sh.am_in[q][k].a);
                const float smin = __uint_as_float(static_cast<unsigned>(sh.am_in[q][rank].b));
                // Messages for row seq + kXchg come only after every pass-2 warp of
                // every CTA is past this row (the rank-0 sender waits for the
                // collector), so the barrier can be re-armed now.
                if (pw == 0 && lane == 0) mbar_arrive_expect_tx(&sh.am_bar[q], kXchgBytes);
                const float m = dec_value(rm);
                // Differences x = l - m below -31 have term 0; they are clamped
                // there (keeps n and the exponent arithmetic in range) unless no
                // logit of the slice needs it. Padding (-inf) clamps to a zero
                // term, so every thread adds exactly ncol terms.
                const bool noclamp = smin - m >= -31.0f;
                const f2 m2 = dup(m);
                unsigned hi = 0, lo = 0;
                const uint32_t tb = sh.tmem + lane_off + static_cast<uint32_t>(t * kRowCols + c0w);
                for (int c0 = 0; c0 < ncol; c0 += 32) {
                    uint32_t rr[32];
                    tmem_ld32(tb + c0, rr);
                    if (noclamp) {
#pragma unroll
                        for (int k = 0; k < 32; k += 2)
                            add_terms(fsub2(pk(__uint_as_float(rr[k]), __uint_as_float(rr[k + 1])), m2),
                                      hi, lo);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            float d0, d1;
                            upk(fsub2(pk(__uint_as_float(rr[k]), __uint_as_float(rr[k + 1])), m2),
                                d0, d1);
                            add_terms(pk(fmaxf(d0, -31.0f), fmaxf(d1, -31.0f)), hi, lo);
                        }
                    }
                }
                tc_fence_before();  // the row's TMEM loads (waited on) before the slot is freed
                hi -= static_cast<unsigned>(ncol) * kMagic43Bits;
                lo -= static_cast<unsigned>(ncol) * kMagic23Bits;
                unsigned long long acc = (static_cast<unsigned long long>(hi) << 20) +
                                         static_cast<long long>(static_cast<int>(lo));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += shfl_xor64(acc, o);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sh.tfree[t]);  // this warp is done with the slot
                    sh.red_sum[q][pw] = acc;
                    if (pw == 0) sh.row_arg[q] = dec_index(rm);
                    mbar_arrive(&sh.p2_done[q]);
                }
            }
        } else if (warp == kAmSenderWarp) {
            // ------------------------------------------------------------ slice sender
            for (int seq = 0; seq < total && ok; ++seq) {
                const int q = seq % kXchg;
                ok = __all_sync(0xffffffffu, mbar_wait(&sh.p1_done[q], (seq / kXchg) & 1, limit));
                if (!ok) break;
                unsigned long long a = lane < kP1Warps ? sh.red_am[q][lane] : 0ull;
                float mnv = lane < kP1Warps ? sh.red_min[q][lane] : INFINITY;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    a = max(a, shfl_xor64(a, o));
                    mnv = fminf(mnv, __shfl_xor_sync(0xffffffffu, mnv, o));
                }
                // CTA 0 reuses exchange slot q only once the collector is done with it.
                if (rank == 0 && seq >= kXchg && lane == 0)
                    ok = mbar_wait(&sh.col_done[q], ((seq / kXchg) - 1) & 1, limit);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane < kCommitCluster)  // lane j sends to CTA j
                    st_async_v2_b64(mapa_shared(smem_u32(&sh.am_in[q][rank]), lane), a,
                                    __float_as_uint(mnv), mapa_shared(smem_u32(&sh.am_bar[q]), lane));
                __syncwarp();
            }
        } else {
            // ------------------------------------------------------------ key sender
            for (int seq = 0; seq < total && ok; ++seq) {
                const int q = seq % kXchg;
                ok = __all_sync(0xffffffffu, mbar_wait(&sh.p2_done[q], (seq / kXchg) & 1, limit));
                if (!ok) break;
                unsigned long long a = lane < kP2Warps ? sh.red_sum[q][lane] : 0ull;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a += shfl_xor64(a, o);
                if (lane == 0)
                    st_async_v2_b64(mapa_shared(smem_u32(&sh.sum_in[q][rank]), 0), a,
                                    rank == 0 ? static_cast<unsigned>(sh.row_arg[q]) : 0u,
                                    mapa_shared(smem_u32(&sh.sum_bar[q]), 0));
                __syncwarp();
            }
        }
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        __syncwarp();
    }
    // No CTA leaves while another may still write into its shared memory.
    tc_fence_before();
    cluster_sync_all();
    // The last cluster to finish puts the call's counters back to zero.
    if (rank == 0 && tid == 0) {
        const unsigned f = atom_add_acq_rel_gpu(p.counters + kCtrFinished, 1u);
        if (f + 1 == static_cast<unsigned>(ncl)) {
            p.counters[kCtrStarted] = 0;
            p.counters[kCtrFinished] = 0;
        }
    }
    // A receiver that gave up may still be the target of a message issued
    // before its sender reached the barrier above: give it 100 us to land
    // before this CTA's shared memory goes away (only after a timeout).
    if (sh.xchg_err) {
        if (tid == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 100000) __nanosleep(1000);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(sh.tmem, 512);
    }
}

}  // namespace

size_t commit_smem_bytes(int /*V*/, int /*L*/) {
    return static_cast<size_t>(kSlots) * kChunk * 4 + static_cast<size_t>(kSelChunk) * 8 +
           2 * (kCommitMaxL / 32) * 4;
}

int commit_max_clusters() {
    // per device, filled on first use; handles on several host threads may ask at once
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    const int known = cached[dev].load(std::memory_order_relaxed);
    if (known > 0) return known;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCommitCluster * 256, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = commit_smem_bytes(kCommitCluster * kCommitSliceMax, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, commit_kernel, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms / kCommitCluster > 0 ? sms / kCommitCluster : 1;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_commit(const CommitParams& p, cudaStream_t s) {
    const long rows = static_cast<long>(p.B) * p.L;
    const int ncl = static_cast<int>(rows < commit_max_clusters() ? rows : commit_max_clusters());
    commit_kernel<<<static_cast<unsigned>(ncl) * kCommitCluster, kThreads,
                    commit_smem_bytes(p.V, p.L), s>>>(p);
    return cudaGetLastError();
}

cudaError_t configure_commit_kernels() {
    return cudaFuncSetAttribute(commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(commit_smem_bytes(kCommitCluster * kCommitSliceMax, 1)));
}

}  // namespace tt
