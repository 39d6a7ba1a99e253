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

// The canonical key and its exponential: commit_key.cuh.
#include <atomic>

#include "commit_key.cuh"
#include "commit_select.cuh"
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

using namespace key;

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
using sel::kSelChunk;                     // keys staged per selection pass
static_assert(kSliceMax == kCommitSliceMax, "slice per CTA");
static_assert(2 * kRowCols == 512, "two row slots fill the TMEM");

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
    __syncthreads();  // the cluster's share (sh.total, sh.row0) is known
    // The producer (lane 0 of its warp): the cluster's masked rows go through
    // the ring in row order, max(nchunks, 1) entries each; the unmasked ones
    // are only marked in masked_out. It issues the first row's entries before
    // the cluster barrier (they use only this CTA's barriers) and the rest once
    // the first entry has landed, so that the first row arrives first.
    const uint64_t pol = l2_policy_evict_first();
    const int per_row = max(nchunks, 1);
    int pr_it = 0, pr_done = 0, pr_r = sh.row0, pr_c = 0;  // entries issued; rows started; row; chunk
    bool pr_ok = true;
    auto produce = [&](int it_end) {
        while (pr_ok && pr_it < it_end) {
            if (pr_c == 0) {
                // next masked row of the share; masked may alias masked_out:
                // this read precedes the block's selection, which waits for
                // this row's ticket
                while (pr_r < rows && __ldcg(p.masked + pr_r) == 0) {
                    if (rank == 0) p.masked_out[pr_r] = 0;
                    ++pr_r;
                }
                if (pr_r >= rows || pr_done == sh.total) return;  // the next cluster's first row
                ++pr_done;
            }
            const int s = pr_it % kSlots;
            if (pr_it >= kSlots && !mbar_wait(&sh.empty[s], ((pr_it / kSlots) - 1) & 1, limit)) {
                pr_ok = false;
                return;
            }
            const int lo = pr_c * kChunk, n = min(kChunk, cnt - lo);
            if (n > 0) {
                mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(n) * 4);
                bulk_load(ring + static_cast<size_t>(s) * kChunk,
                          p.logits + static_cast<size_t>(pr_r) * p.V + v0 + lo, static_cast<uint32_t>(n) * 4,
                          &sh.full[s], pol);
            } else {
                mbar_arrive(&sh.full[s]);
            }
            ++pr_it;
            if (++pr_c == per_row) {
                pr_c = 0;
                ++pr_r;
            }
        }
    };
    if (warp == kProducerWarp && lane == 0) produce(per_row);
    tc_fence_before();
    // Every CTA's barriers are initialised before any remote arrival.
    cluster_sync_all();
    tc_fence_after();
    // The cluster's scans are over. When masked_out is the masked buffer, no
    // block selection writes the mask before every cluster has scanned it (the
    // selecting warp waits for this count to reach the number of clusters).
    // (Counted by a warp that is idle until the first row's exchange.)
    if (rank == 0 && warp == kSumSenderWarp && lane == 0) red_add_release_gpu(p.counters + kCtrStarted, 1u);

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            if (pr_it > 0 && !mbar_wait(&sh.full[0], 0, limit)) pr_ok = false;
            produce(0x7fffffff);
            if (!pr_ok) atomicOr(p.status, kDevWaitTimeout);
            // Let the copies already issued land before the CTA can exit (an
            // entry is issued only once the one kSlots before it was consumed, so
            // at most the last kSlots can be in flight; after a normal run they
            // have all landed). Also when a consumer gave up instead.
            const uint64_t dl = drain_limit(limit);
            for (int j = pr_it - kSlots < 0 ? 0 : pr_it - kSlots; j < pr_it; ++j)
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
                    if (p.L <= 32 * sel::kSelRegRows) sel::select_block_small(p, cb, cnum, lane);
                    else sel::select_block(p, cb, cnum, s_key, s_mbits, s_cbits, lane);
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
                // The warp's sum of (hi << 20) + lo with 32-bit warp reductions:
                // per lane 0 <= hi < 2^28 and |lo| <= ncol * 2^19 <= 2^26, so
                // 16-bit halves of hi and of lo + 2^26 sum over 32 lanes
                // without overflow.
                const unsigned lo_u = lo + (1u << 26);
                const unsigned h0 = __reduce_add_sync(0xffffffffu, hi & 0xFFFFu);
                const unsigned h1 = __reduce_add_sync(0xffffffffu, hi >> 16);
                const unsigned l0 = __reduce_add_sync(0xffffffffu, lo_u & 0xFFFFu);
                const unsigned l1 = __reduce_add_sync(0xffffffffu, lo_u >> 16);
                const unsigned long long acc =
                    (((static_cast<unsigned long long>(h1) << 16) + h0) << 20) +
                    ((static_cast<unsigned long long>(l1) << 16) + l0) - (32ull << 26);
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
