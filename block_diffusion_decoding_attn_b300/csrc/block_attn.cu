// Block attention of the TwoTower denoiser ("Nemotron-Labs-TwoTower",
// Section 2.1, Eq. 1): every query of the L-token noisy block takes one
// softmax over [context-tower keys 0..ctx_len-1 of this layer; the block's own
// L keys], with no mask inside the block and GQA head sharing.
//
// The causal variant (p.causal) is the context tower's pass over a committed
// block (Section 2.1, Algorithm 1, the context update after a commit): block
// query l sees the context and block keys 0..l only. The block tiles are
// masked per row; a row with no visible key in a piece of its keys (a block
// tile past it) keeps m = -inf, a zero sum and zero P there, and the merge
// gives such a piece weight 0.
//
// The batched training layout (p.ctx_group = n, Section 2.3, "Implementation":
// all noisy blocks of a clean sequence in one pass, each attending to the past
// clean blocks and bidirectionally within itself) is the same computation
// over B*n sequences of L = S tokens: sequence b is noisy block b % n of clean
// sequence b / n, reads that sequence's cache and sees its first (b % n) * S
// positions.
//
// Work decomposition. The G = Hq/Hkv query heads of a KV head are packed with
// the block positions into the M dimension (row = l*G + g); a CTA computes two
// 128-row query tiles (a pair) against one KV tile at a time, so each K/V tile
// staged in shared memory feeds 256 query rows. The kernel is persistent: one
// CTA per SM, in groups of `width` CTAs. The pairs of a (b, KV head) are cut
// into pair blocks of `width`; a unit is (b, KV head, pair block) with the
// sequence's ctx_len/128 + L/128 KV tiles (rounded up). Every CTA reads the
// lengths and lays the units' tiles end to end (sequence, KV head, pair block,
// tile); the line is cut into one contiguous range per group (stream-K), so
// every group gets the same number of tiles whatever the mix of lengths. CTA j
// of a group takes pair j of each unit in its range: the width CTAs of a group
// read the same K/V tiles at the same time (one HBM read, the rest from L2).
// A query tile whose tiles were cut between groups is finished by the group
// that completes it last: every piece writes its partial (running max, running
// sum, unnormalised O), takes a ticket, and the last one merges the pieces in
// group order (deterministic) and writes the output.
//
// Warp roles (320 threads):
//   warps 0-3  softmax of query tile A, warps 4-7 of tile B: one query row per
//              thread; S from TMEM, online softmax in fp32 (log2 domain), P as
//              bf16 back into TMEM over the first half of S; rescales O in TMEM
//              when the running max grows by more than 2^8; epilogue of each
//              unit (output, or partial + ticket + merge)
//   warp 8     TMA producer: the pair's Q tiles per unit (as soon as the last
//              QK^T of the previous unit has completed), K_j, V_j into a
//              5-slot ring
//   warp 9     MMA issuer (tcgen05, fp32 accumulators in TMEM) and TMEM owner
// TMEM columns: S_A 0-127, O_A 128-255, S_B 256-383, O_B 384-511. P_X lives in
// columns 0-63 of S_X (two bf16 per column) and is the A operand of O_X += P V.
// The tensor core runs the two tiles in ping-pong: while tile A's softmax runs
// it computes tile B's P V and next S, and the other way round. tcgen05.mma
// operations complete in issue order, so "S_X(j) complete" also means
// "P V of tile X for KV tile j-1 complete": the softmax may then overwrite S_X
// with P and rescale O_X without another wait. The MMA warp waits on one
// barrier per group: P_X complete also means the group's V_j and K_j+1 have
// landed (tile A's softmax waits for them before it signals) and, on a unit's
// first tile, that the previous unit's O_X has been read out (each softmax
// thread signals that before it can signal the next unit's P).
#include "ptx.cuh"
#include "tt_internal.h"

namespace tt {

namespace {

constexpr int kRing = 5;               // K/V tile slots (K_j and V_j alternate)
constexpr float kRescaleThresh = 8.0f; // log2 units
constexpr int kThreads = 320;

template <int D>
struct AttnLayout {
    static constexpr int kTileBytes = kTile * D * 2;  // a Q, K or V tile (bf16)
    static constexpr int kAtomBytes = kTile * 128;    // one 64-column swizzle atom column
    static constexpr int kQ = 0;                      // Q_A, then Q_B
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBar = kRingOff + kRing * kTileBytes;
    // q_full, q_empty, full[kRing], empty[kRing], s_full[2], p_full[2],
    // o_final[2], o_empty[2], drain
    static constexpr int kNumBars = 2 + 2 * kRing + 9;
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

// ctx_len of sequence b (clamped to [0, ctx_cap]; *bad set if it was outside)
// and its number of KV tiles (context tiles, then block tiles).
__device__ __forceinline__ int seq_tiles(const AttnParams& p, int b, int& C, bool& bad) {
    C = p.ctx_group ? (b % p.ctx_group) * p.L : __ldg(p.ctx_len + b);
    if (C < 0 || C > p.ctx_cap) {
        bad = true;
        C = C < 0 ? 0 : p.ctx_cap;
    }
    return (C + kTile - 1) / kTile + p.nblk;
}

// One contiguous piece of a unit's KV tiles, as every role of the CTA walks
// them (the same sequence of items in every role). On the line a unit takes
// its KV tiles plus p.item_cost positions that hold no tile (the fixed cost of
// a unit: loading Q, starting the pipeline, the epilogue), so that the cut
// balances work rather than tile counts.
struct Item {
    int b, kvh, pq;       // the unit: sequence, KV head, pair block
    int C, tiles;         // ctx_len of b (clamped) and its KV tiles
    long long pb;         // line position of sequence b's first unit
    long long ustart;     // line position of this unit's first tile
    int t0, t1;           // this item's tiles [t0, t1) of the unit
};

struct Sched {
    long long T;   // positions on the line
    int geff;      // groups with work
    long long s, e;  // this group's range
    int b;         // sequence holding position s
    long long pb;  // line position of its first unit
};

__device__ __forceinline__ long long grp_start(long long g, long long T, int geff) {
    return g * T / geff;
}
// The group whose range holds line position x.
__device__ __forceinline__ int grp_of(long long x, long long T, int geff) {
    return static_cast<int>(((x + 1) * geff - 1) / T);
}

// The unit after `it` on the line (sequence, KV head, pair block order).
__device__ __forceinline__ void advance_unit(const AttnParams& p, Item& it) {
    const int nq = p.n_pairs / p.width;
    it.ustart += it.tiles + p.item_cost;
    if (++it.pq == nq) {
        it.pq = 0;
        if (++it.kvh == p.Hkv) {
            it.kvh = 0;
            it.pb += static_cast<long long>(it.tiles + p.item_cost) * p.Hkv * nq;
            ++it.b;
            bool bad = false;
            it.tiles = seq_tiles(p, it.b, it.C, bad);
        }
    }
}

// The group's first item (a range is longer than a unit's tail of
// item_cost positions, so it holds at least one tile).
__device__ __forceinline__ Item first_item(const AttnParams& p, const Sched& sc) {
    const int nq = p.n_pairs / p.width;
    Item it;
    bool bad = false;
    it.b = sc.b;
    it.pb = sc.pb;
    it.tiles = seq_tiles(p, it.b, it.C, bad);
    const long long u = (sc.s - sc.pb) / (it.tiles + p.item_cost);
    it.kvh = static_cast<int>(u / nq);
    it.pq = static_cast<int>(u % nq);
    it.ustart = sc.pb + u * (it.tiles + p.item_cost);
    long long t0 = sc.s - it.ustart;
    if (t0 >= it.tiles) {  // the range starts in a unit's tail: the next unit
        advance_unit(p, it);
        t0 = 0;
    }
    it.t0 = static_cast<int>(t0);
    it.t1 = static_cast<int>(min(static_cast<long long>(it.tiles), sc.e - it.ustart));
    return it;
}

// Moves to the group's next item; false when the range is done.
__device__ __forceinline__ bool next_item(const AttnParams& p, const Sched& sc, Item& it) {
    if (it.ustart + it.tiles + p.item_cost >= sc.e) return false;
    advance_unit(p, it);
    it.t0 = 0;
    it.t1 = static_cast<int>(min(static_cast<long long>(it.tiles), sc.e - it.ustart));
    return true;
}

// Barrier among the 128 softmax threads of one query tile (ids 1 and 2; 0 is
// __syncthreads).
template <int kId>
__device__ __forceinline__ void tile_bar() {
    asm volatile("bar.sync %0, 128;" ::"n"(kId) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* a, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}

template <int D>
__device__ __forceinline__ void store_out_row(const AttnParams& p, int b, int kvh, int m,
                                              const float* o, float inv) {
    const int l = m / p.G, g = m % p.G;
    __nv_bfloat16* dst = p.out + ((static_cast<size_t>(b) * p.L + l) * p.Hq + kvh * p.G + g) * D;
#pragma unroll
    for (int c = 0; c < D; c += 8) {
        const uint4 v = make_uint4(pack_bf16x2(o[c] * inv, o[c + 1] * inv),
                                   pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv),
                                   pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv),
                                   pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv));
        *reinterpret_cast<uint4*>(dst + c) = v;
    }
}


__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// One query tile's piece of a unit cut between groups (O still in TMEM at
// `to`, this thread's row; running max m_run and sum l_run). Writes the
// partial (O in 32-column chunks straight from TMEM, then max and sum), takes
// the tile's ticket with one release per tile, and if it is the last piece
// merges all pieces in group order and stores the output row. The caller
// frees O's TMEM afterwards.
template <int D>
__device__ __noinline__ void epilogue_piece(const AttnParams& p, const Sched& sc, const Item& it,
                                            int x, int row, int m, bool live, int grp, int pj,
                                            uint32_t to, float m_run, float l_run, int* sh_last) {
    constexpr int kQ = D / 32;  // 32-column chunks of a row
    const int mt = 2 * (it.pq * p.width + pj) + x;
    // A CTA's range cuts at most two of its units: one that it starts in the
    // middle (slot 0) and one that it starts at tile 0 and does not finish
    // (slot 1).
    const size_t slot = 2 * static_cast<size_t>(blockIdx.x) + (it.t0 == 0 ? 1 : 0);
    float4* po = reinterpret_cast<float4*>(p.part_o + (slot * 2 + x) * (kTile * D));
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
        uint32_t r[32];
        tmem_ld32(to + q * 32, r);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
            __stcg(po + (q * 8 + c4) * kTile + row,
                   make_float4(__uint_as_float(r[4 * c4]), __uint_as_float(r[4 * c4 + 1]),
                               __uint_as_float(r[4 * c4 + 2]), __uint_as_float(r[4 * c4 + 3])));
    }
    __stcg(p.part_ml + (slot * 2 + x) * kTile + row, make_float2(m_run, l_run));
    const int i0 = grp_of(it.ustart, sc.T, sc.geff);
    const int i1 = grp_of(it.ustart + it.tiles - 1, sc.T, sc.geff);
    // every thread's stores, then one release with the ticket
    if (x) tile_bar<2>(); else tile_bar<1>();
    if (row == 0) {
        unsigned* tk = p.tickets + (static_cast<size_t>(it.b) * p.Hkv + it.kvh) * p.n_mtiles + mt;
        fence_acq_rel_gpu();
        const unsigned t = atom_add_acq_rel(tk, 1u);
        const int last = t + 1 == static_cast<unsigned>(i1 - i0 + 1);
        if (last) *tk = 0u;  // no other ticket of this call remains
        *sh_last = last;
    }
    if (x) tile_bar<2>(); else tile_bar<1>();
    if (!*sh_last) return;
    fence_acq_rel_gpu();
    // Group g's piece starts in the middle of the unit (slot 0) unless g = i0,
    // whose range holds the unit's first tile (slot 1).
    auto slot_of = [&](int g) { return static_cast<size_t>(2 * (g * p.width + pj) + (g == i0 ? 1 : 0)); };
    const int l = m / p.G, g_head = m % p.G;
    __nv_bfloat16* dst = p.out + ((static_cast<size_t>(it.b) * p.L + l) * p.Hq + it.kvh * p.G + g_head) * D;
    if (i1 == i0 + 1) {
        // Two pieces: this one from TMEM, the other from its partial. Products
        // and the sum are rounded separately, in group order, so either piece
        // computes the same bits.
        const bool mine_first = grp == i0;
        const size_t so = slot_of(mine_first ? i1 : i0);
        const float2 ml = __ldcg(p.part_ml + (so * 2 + x) * kTile + row);
        const float m1 = mine_first ? m_run : ml.x, m2 = mine_first ? ml.x : m_run;
        const float l1 = mine_first ? l_run : ml.y, l2 = mine_first ? ml.y : l_run;
        const float mx = fmaxf(m1, m2);
        const float w1 = ex2_approx(m1 - mx), w2 = ex2_approx(m2 - mx);  // 0: a piece with no visible key
        const float wm = mine_first ? w1 : w2, wo = mine_first ? w2 : w1;
        const float inv = 1.f / __fadd_rn(__fmul_rn(w1, l1), __fmul_rn(w2, l2));
        const float4* src = reinterpret_cast<const float4*>(p.part_o + (so * 2 + x) * (kTile * D));
        float4 nxt[8];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) nxt[c4] = __ldcg(src + c4 * kTile + row);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            float4 cur[8];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) cur[c4] = nxt[c4];
            if (q + 1 < kQ) {
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) nxt[c4] = __ldcg(src + ((q + 1) * 8 + c4) * kTile + row);
            }
            uint32_t r[32];
            tmem_ld32(to + q * 32, r);
            uint32_t pk[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float ov[4] = {cur[c4].x, cur[c4].y, cur[c4].z, cur[c4].w};
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = __fmul_rn(wm, __uint_as_float(r[4 * c4 + e])), b = __fmul_rn(wo, ov[e]);
                    v[e] = (mine_first ? __fadd_rn(a, b) : __fadd_rn(b, a)) * inv;
                }
                pk[2 * c4] = pack_bf16x2(v[0], v[1]);
                pk[2 * c4 + 1] = pack_bf16x2(v[2], v[3]);
            }
            if (live) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(dst + q * 32 + u * 8) =
                        make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
        }
    } else {
        // More pieces: every piece (this one too) from its partial, in group order.
        float mx = -INFINITY;
        for (int g = i0; g <= i1; ++g)
            mx = fmaxf(mx, __ldcg(p.part_ml + (slot_of(g) * 2 + x) * kTile + row).x);
        float den = 0.f;
        for (int g = i0; g <= i1; ++g) {
            const float2 ml = __ldcg(p.part_ml + (slot_of(g) * 2 + x) * kTile + row);
            den = __fadd_rn(den, __fmul_rn(ex2_approx(ml.x - mx), ml.y));
        }
        const float inv = 1.f / den;
#pragma unroll 1
        for (int q = 0; q < kQ; ++q) {
            float acc[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 1
            for (int g = i0; g <= i1; ++g) {
                const size_t sl = slot_of(g);
                const float wgt = ex2_approx(__ldcg(p.part_ml + (sl * 2 + x) * kTile + row).x - mx);
                const float4* src = reinterpret_cast<const float4*>(p.part_o + (sl * 2 + x) * (kTile * D));
                float4 v[8];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) v[c4] = __ldcg(src + (q * 8 + c4) * kTile + row);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    acc[4 * c4] = __fadd_rn(acc[4 * c4], __fmul_rn(wgt, v[c4].x));
                    acc[4 * c4 + 1] = __fadd_rn(acc[4 * c4 + 1], __fmul_rn(wgt, v[c4].y));
                    acc[4 * c4 + 2] = __fadd_rn(acc[4 * c4 + 2], __fmul_rn(wgt, v[c4].z));
                    acc[4 * c4 + 3] = __fadd_rn(acc[4 * c4 + 3], __fmul_rn(wgt, v[c4].w));
                }
            }
            if (live) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(dst + q * 32 + u * 8) = make_uint4(
                        pack_bf16x2(acc[8 * u] * inv, acc[8 * u + 1] * inv),
                        pack_bf16x2(acc[8 * u + 2] * inv, acc[8 * u + 3] * inv),
                        pack_bf16x2(acc[8 * u + 4] * inv, acc[8 * u + 5] * inv),
                        pack_bf16x2(acc[8 * u + 6] * inv, acc[8 * u + 7] * inv));
            }
        }
    }
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    block_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_kc,
                      const __grid_constant__ CUtensorMap tm_vc,
                      const __grid_constant__ CUtensorMap tm_kb,
                      const __grid_constant__ CUtensorMap tm_vb, const AttnParams p) {
    using Lay = AttnLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ long long sh_wsum[kThreads / 32];
    __shared__ int sh_umin[kThreads / 32], sh_umax[kThreads / 32];
    __shared__ int sh_b;
    __shared__ long long sh_pb;
    __shared__ int sh_last[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = blockIdx.x / p.width;
    const int pj = blockIdx.x % p.width;  // pair of each unit's pair block taken by this CTA

    if (warp == 8 && lane == 0) {  // descriptor fetches overlap the schedule scan
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kc);
        tma_prefetch_desc(&tm_vc);
        tma_prefetch_desc(&tm_kb);
        tma_prefetch_desc(&tm_vb);
    }

    // ------------------------------------------------------------ schedule
    // Tiles per sequence, a block-wide scan over the sequences, and the
    // sequence that holds the start of this group's range.
    Sched sc;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::kBar);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* full = bars + 2;
    uint64_t* empty = full + kRing;
    uint64_t* s_full = empty + kRing;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_final = p_full + 2;
    uint64_t* o_empty = o_final + 2;
    uint64_t* drain = o_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Lay::kTmemSlot);
    {
        const long long mult = static_cast<long long>(p.Hkv) * (p.n_pairs / p.width);
        const int per = (p.B + kThreads - 1) / kThreads;
        const int b_lo = min(p.B, tid * per), b_hi = min(p.B, b_lo + per);
        long long sum = 0;
        bool bad = false;
        int umin = 0x7fffffff, umax = 0;  // unit lengths on the line
        for (int b = b_lo; b < b_hi; ++b) {
            int C;
            const int ul = seq_tiles(p, b, C, bad) + p.item_cost;
            sum += ul * mult;
            umin = min(umin, ul);
            umax = max(umax, ul);
        }
        if (bad && blockIdx.x == 0) atomicOr(p.status, kDevCtxLenRange);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            umin = min(umin, __shfl_xor_sync(0xffffffffu, umin, o));
            umax = max(umax, __shfl_xor_sync(0xffffffffu, umax, o));
        }
        if (lane == 0) {
            sh_umin[warp] = umin;
            sh_umax[warp] = umax;
        }
        long long inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) sh_wsum[warp] = inc;
        __syncthreads();
        long long wpre = 0, T = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const long long v = sh_wsum[w];
            T += v;
            wpre += w < warp ? v : 0;
            umin = min(umin, sh_umin[w]);
            umax = max(umax, sh_umax[w]);
        }
        sc.T = T;
        const long long g_max = T / p.min_tiles;
        sc.geff = static_cast<int>(min(static_cast<long long>(p.ngroups), g_max < 1 ? 1 : g_max));
        // Units of one length: whole units per group, k each, when that is no
        // slower than cutting (the line cut evenly, plus a cut's cost).
        if (umin == umax) {
            const long long units = T / umin;
            const long long k = (units + p.ngroups - 1) / p.ngroups;
            if (units % k == 0 && k * umin <= T / p.ngroups + p.cut_cost)
                sc.geff = static_cast<int>(units / k);
        }
        if (grp >= sc.geff) return;  // no work for this group (uniform over the CTA)
        // barriers and tensor memory while one thread finds the range's start
        if (tid == 0) {
            mbar_init(q_full, 1);
            mbar_init(q_empty, 1);
            for (int s = 0; s < kRing; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(&s_full[s], 1);
                mbar_init(&p_full[s], 128);
                mbar_init(&o_final[s], 1);
                mbar_init(&o_empty[s], 128);
            }
            mbar_init(drain, 1);
            fence_mbar_init();
        }
        if (warp == 9) {
            tmem_alloc(tmem_slot, 512);
            tmem_relinquish();
        }
        sc.s = grp_start(grp, T, sc.geff);
        sc.e = grp_start(grp + 1, T, sc.geff);
        const long long excl = wpre + inc - sum;
        if (sum > 0 && excl <= sc.s && sc.s < excl + sum) {
            long long pos = excl;
            for (int b = b_lo; b < b_hi; ++b) {
                int C;
                const long long wb = (seq_tiles(p, b, C, bad) + p.item_cost) * mult;
                if (sc.s < pos + wb) {
                    sh_b = b;
                    sh_pb = pos;
                    break;
                }
                pos += wb;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    sc.b = sh_b;
    sc.pb = sh_pb;
    const uint32_t tmem = *tmem_slot;
    const uint64_t limit = p.timeout_ns;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int rows_l = kTile / p.G;  // block positions per query tile
            bool ok = true;
            int li = 0;   // ring loads issued: K_j is load 2j, V_j is load 2j+1 (j over all items)
            int nit = 0;  // units whose Q was issued
            Item it = first_item(p, sc);
            do {
                // Q_A, Q_B of this unit once the previous unit's last QK^T has completed.
                if (nit > 0 && !mbar_wait(q_empty, (nit - 1) & 1, limit)) { ok = false; break; }
                const int pair = it.pq * p.width + pj;
                mbar_arrive_expect_tx(q_full, 2 * Lay::kTileBytes);
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_5d(sm + Lay::kQ + t * Lay::kTileBytes + c * Lay::kAtomBytes, &tm_q,
                                    q_full, c * 64, 0, it.kvh, (2 * pair + t) * rows_l, it.b);
                ++nit;
                {
                    // the next unit's Q into L2 now: its load waits for this
                    // unit's last QK^T, and then comes from L2
                    Item nx = it;
                    if (next_item(p, sc, nx)) {
                        const int npair = nx.pq * p.width + pj;
#pragma unroll
                        for (int t = 0; t < 2; ++t)
#pragma unroll
                            for (int c = 0; c < D / 64; ++c)
                                tma_prefetch_5d(&tm_q, c * 64, 0, nx.kvh, (2 * npair + t) * rows_l, nx.b);
                    }
                }
                const int nc = (it.C + kTile - 1) / kTile;
                const int cache_row = (p.ctx_group ? it.b / p.ctx_group : it.b) * p.Hkv + it.kvh;
                for (int j = it.t0; j < it.t1 && ok; ++j) {
                    const KvTile t = kv_tile(j, nc, it.C, p.L);
#pragma unroll 1
                    for (int kv = 0; kv < 2; ++kv, ++li) {
                        const int slot = li % kRing;
                        if (li >= kRing && !mbar_wait(&empty[slot], ((li / kRing) & 1) ^ 1, limit)) {
                            ok = false;
                            break;
                        }
                        uint8_t* dst = sm + Lay::kRingOff + slot * Lay::kTileBytes;
                        mbar_arrive_expect_tx(&full[slot], Lay::kTileBytes);
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) {
                            if (t.is_ctx)
                                tma_load_3d(dst + c * Lay::kAtomBytes, kv ? &tm_vc : &tm_kc,
                                            &full[slot], c * 64, t.base, cache_row);
                            else
                                tma_load_4d(dst + c * Lay::kAtomBytes, kv ? &tm_vb : &tm_kb,
                                            &full[slot], c * 64, it.kvh, t.base, it.b);
                        }
                    }
                }
            } while (ok && next_item(p, sc, it));
            if (!ok) atomicOr(p.status, kDevWaitTimeout);
            // Let the copies already issued land before the CTA can exit (a
            // ring load is issued only once the load kRing before it was
            // consumed, so at most the last kRing can be in flight; a unit's Q
            // only after the previous unit's). Also after a timeout of
            // another role.
            const uint64_t dl = drain_limit(limit);
            if (nit > 0) mbar_wait(q_full, (nit - 1) & 1, dl);
            for (int l = li - kRing < 0 ? 0 : li - kRing; l < li; ++l)
                mbar_wait(&full[l % kRing], (l / kRing) & 1, dl);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16(kTile, kTile, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, 0, 1);
        const uint32_t sq = smem_u32(sm + Lay::kQ);
        const uint32_t ring = smem_u32(sm + Lay::kRingOff);
        const uint32_t col_s[2] = {0u, 2u * kTile};
        const uint32_t col_o[2] = {static_cast<uint32_t>(kTile), 3u * kTile};
        auto wait_slot = [&](int l) { return mbar_wait(&full[l % kRing], (l / kRing) & 1, limit); };
        // S_X = Q_X K^T for the K tile in ring load l
        auto issue_s = [&](int x, int l) {
            const uint32_t sk = ring + (l % kRing) * Lay::kTileBytes;
            const uint32_t sqx = sq + x * Lay::kTileBytes;
    #pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * Lay::kAtomBytes + (kk & 3) * 32;
                tc_mma_ss(tmem + col_s[x], sdesc_sw128(sqx + off, 16, 1024),
                          sdesc_sw128(sk + off, 16, 1024), idesc_qk, kk > 0);
            }
        };
        // O_X (+)= P_X V for the V tile in ring load l
        auto issue_pv = [&](int x, int l, bool first) {
            const uint32_t sv = ring + (l % kRing) * Lay::kTileBytes;
    #pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
                // V is MN-major (d contiguous): 16 keys = two 8-row atoms; the
                // next 64 columns of d sit one atom column further.
                const uint64_t bd = sdesc_sw128(sv + kk * 2048, Lay::kAtomBytes, 1024);
                tc_mma_ts(tmem + col_o[x], tmem + col_s[x] + kk * 8, bd, idesc_pv,
                          (!first || kk > 0) ? 1u : 0u);
            }
        };
        // Cache rows past ctx_len may hold anything (even NaN); P is 0 there,
        // but 0 * NaN is not, so zero those V rows of the last context tile.
        auto zero_tail = [&](const KvTile& kt, int l) {
            if (kt.is_ctx && kt.valid < kTile) {
                uint8_t* sv = sm + Lay::kRingOff + (l % kRing) * Lay::kTileBytes;
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

        bool ok = true;
        int gt = 0;   // KV tiles processed over all items (ring load 2 gt = K, 2 gt + 1 = V)
        int nit = 0;  // items started
        Item it = first_item(p, sc);
        do {
            const int n = it.t1 - it.t0;
            const int nc = (it.C + kTile - 1) / kTile;
            ok = mbar_wait(q_full, nit & 1, limit) && wait_slot(2 * gt);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                issue_s(0, 2 * gt);
                tc_commit(&s_full[0]);
                issue_s(1, 2 * gt);
                tc_commit(&s_full[1]);
                tc_commit(&empty[(2 * gt) % kRing]);
                if (n == 1) tc_commit(q_empty);  // the unit's last QK^T is issued
            }
            __syncwarp();
            for (int j = 0; j < n && ok; ++j, ++gt) {
                const int lv = 2 * gt + 1, lk = 2 * gt + 2;
                const bool more = j + 1 < n;
                // ---- tile A: P_A complete also means V_j and K_j+1 have landed
                // (tile A's softmax waits for them before it signals) and, on a
                // unit's first tile, that the previous unit's O_A has been read
                // out (each softmax thread signals that first); one wait, so
                // that the group follows the previous one without a gap
                if (!mbar_wait(&p_full[0], gt & 1, limit)) {
                    ok = false;
                    break;
                }
                zero_tail(kv_tile(it.t0 + j, nc, it.C, p.L), lv);
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
                // ---- tile B (its inputs are tile A's, already in)
                if (!mbar_wait(&p_full[1], gt & 1, limit)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    issue_pv(1, lv, j == 0);
                    tc_commit(&empty[lv % kRing]);
                    if (more) {
                        issue_s(1, lk);
                        tc_commit(&s_full[1]);
                        tc_commit(&empty[lk % kRing]);
                        if (j + 2 == n) tc_commit(q_empty);  // the unit's last QK^T is issued
                    } else {
                        tc_commit(&o_final[1]);
                    }
                }
                __syncwarp();
            }
            ++nit;
        } while (ok && next_item(p, sc, it));
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
        // No MMA may still be running when the TMEM is released.
        if (lane == 0) tc_commit(drain);
        __syncwarp();
        mbar_wait(drain, 0, drain_limit(limit));
    } else {
        // ------------------------------------------------------------ softmax
        const int x = warp >> 2;                 // query tile of the pair
        const int row = (warp & 3) * 32 + lane;  // TMEM lane = row of the tile
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t ts = tmem + lane_off + (x ? 2u * kTile : 0u);
        const uint32_t to = tmem + lane_off + (x ? 3u * kTile : static_cast<uint32_t>(kTile));
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gt = 0, nit = 0;
        Item it = first_item(p, sc);
        do {
            const int n = it.t1 - it.t0;
            const int nc = (it.C + kTile - 1) / kTile;
            const int mt = 2 * (it.pq * p.width + pj) + x;  // query tile of (b, kv head)
            const int m = mt * kTile + row;                 // packed query row
            const int lq = m / p.G;                         // its block position
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < n; ++j, ++gt) {
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], gt & 1, limit));
                if (!ok) break;
                tc_fence_after();
                float s[kTile];
                {
                    uint32_t r[kTile];
                    tmem_ld128(ts, r);
        #pragma unroll
                    for (int c = 0; c < kTile; ++c) s[c] = __uint_as_float(r[c]);
                }
                const KvTile kt = kv_tile(it.t0 + j, nc, it.C, p.L);
                // keys of this tile the row sees: the tile's keys, and in the
                // causal variant only block keys up to the row's own position
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
                if (x == 0 && row == 0) {
                    // the MMA group this P starts reads V_j and K_j+1: have them in first
                    const int lv = 2 * gt + 1, lk = lv + 1;
                    if (!mbar_wait(&full[lv % kRing], (lv / kRing) & 1, limit) ||
                        (j + 1 < n && !mbar_wait(&full[lk % kRing], (lk / kRing) & 1, limit)))
                        atomicOr(p.status, kDevWaitTimeout);
                }
                tc_fence_before();
                mbar_arrive(&p_full[x]);
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_final[x], nit & 1, limit));
            if (!ok) break;
            // ---- epilogue of the unit
            tc_fence_after();
            const bool live = lq < p.L;
            if (it.t0 == 0 && it.t1 == it.tiles) {
                // the whole unit: O out of TMEM (the TMEM is then free), normalise, store
                float o[D];
                {
                    uint32_t r[kTile];
                    tmem_ld128(to, r);  // O (the first D columns)
#pragma unroll
                    for (int c = 0; c < D; ++c) o[c] = __uint_as_float(r[c]);
                }
                tc_fence_before();
                mbar_arrive(&o_empty[x]);
                if (live) store_out_row<D>(p, it.b, it.kvh, m, o, 1.f / l_run);
            } else {
                if (mt < p.n_mtiles) epilogue_piece<D>(p, sc, it, x, row, m, live, grp, pj, to, m_run,
                                                       l_run, &sh_last[x]);
                tc_fence_before();
                mbar_arrive(&o_empty[x]);
            }
            ++nit;
        } while (next_item(p, sc, it));
        if (!ok && lane == 0) atomicOr(p.status, kDevWaitTimeout);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_attn_impl(const AttnMaps& m, const AttnParams& p, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(p.ngroups * p.width), 1, 1);
    block_attn_kernel<D><<<grid, kThreads, AttnLayout<D>::kAlloc, s>>>(m.q, m.k_ctx, m.v_ctx,
                                                                      m.k_blk, m.v_blk, p);
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

cudaError_t launch_block_attn(const AttnMaps& maps, const AttnParams& p, int D, cudaStream_t s) {
    return D == 64 ? launch_attn_impl<64>(maps, p, s) : launch_attn_impl<128>(maps, p, s);
}

}  // namespace tt
