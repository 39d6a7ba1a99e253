// Internal interface between the C-ABI layer (tt_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace tt {

// Device status bits (accumulated in the handle's status word).
constexpr unsigned kDevCtxLenRange = 1u;  // ctx_len[b] outside [0, ctx_cap]; clamped
constexpr unsigned kDevWaitTimeout = 2u;  // a bounded pipeline wait gave up
// Bound of the waits for work a CTA issued itself (its TMA copies, its MMAs)
// before it leaves, whatever the pipeline wait limit: that work always
// completes, and the CTA's shared and tensor memory must outlive it.
constexpr unsigned long long kDrainNs = 100000000ull;  // 100 ms
__host__ __device__ inline unsigned long long drain_limit(unsigned long long limit) {
    return limit > kDrainNs ? limit : kDrainNs;
}

constexpr int kTile = 128;  // query rows per M tile and keys per KV tile

struct AttnParams {
    int B, L, Hq, Hkv, G, ctx_cap;
    int n_mtiles;  // ceil(G*L / 128) query tiles per (b, kv head)
    int n_pairs;   // ceil(n_mtiles / 2): a CTA takes two query tiles at a time
    int nblk;      // ceil(L / 128) tiles of block keys
    int causal;    // 1: block query l sees block keys 0..l only (context-tower update)
    // Batched training layout (0: off). Sequence b is noisy block b % ctx_group
    // of clean sequence b / ctx_group: it reads that sequence's cache, with
    // ctx_len = (b % ctx_group) * L (ctx_len is then not read).
    int ctx_group;
    // Persistent schedule: the grid is `ngroups` groups of `width` CTAs. The
    // n_pairs query-tile pairs of a (b, kv head) are cut into n_pairs / width
    // pair blocks; a work unit of a group is (b, kv head, pair block) over the
    // sequence's KV tiles, CTA j of the group taking pair j of the block. The
    // units' KV tiles are laid end to end and cut into one contiguous range per
    // group (at least min_tiles tiles each; groups past the work exit).
    int width, ngroups, min_tiles;
    int item_cost;  // line positions a unit takes beyond its tiles (< min_tiles)
    int cut_cost;   // line positions a cut unit costs (partial out, ticket, merge)
    float scale_log2;
    const int32_t* ctx_len;
    __nv_bfloat16* out;
    // Partial results of a query tile whose KV tiles were cut between groups:
    // two slots per CTA (its first and its last unit), each holding both query
    // tiles: O as [2][D/4][128][4] fp32 and (running max, running sum) as
    // [2][128] float2.
    float* part_o;
    float2* part_ml;
    // One counter per query tile (B * Hkv * n_mtiles): the pieces of a cut
    // tile take a ticket after writing their partial; the last one merges and
    // puts the counter back to zero. Zero between calls.
    unsigned* tickets;
    unsigned* status;
    unsigned long long timeout_ns;
};

// The one-unit-per-CTA schedule (block_attn_split.cu): one CTA per (b, KV
// head, query-tile pair, KV split of `chunk` tiles).
struct AttnSplitParams {
    int B, L, Hq, Hkv, G, ctx_cap;
    int n_mtiles, n_pairs, nblk, causal, ctx_group;
    int chunk;     // KV tiles per split
    float scale_log2;
    const int32_t* ctx_len;
    __nv_bfloat16* out;
    float* ws_o;   // split partials [splits][B][Hkv][n_mtiles*128][D] (nullptr: one split)
    float* ws_ml;  // [splits][B][Hkv][n_mtiles*128][2] = (running max, running sum)
    unsigned* status;
    unsigned long long timeout_ns;
};

struct AttnMaps {
    CUtensorMap q, k_ctx, v_ctx, k_blk, v_blk;
};

// Partial-result bytes of one CTA slot for head dim D (both query tiles).
constexpr size_t attn_slot_o_floats(int D) { return static_cast<size_t>(2) * kTile * D; }
constexpr size_t attn_slot_ml(int /*D*/) { return static_cast<size_t>(2) * kTile; }

cudaError_t launch_block_attn(const AttnMaps& maps, const AttnParams& p, int D, cudaStream_t s);
cudaError_t launch_block_attn_split(const AttnMaps& maps, const AttnSplitParams& p, int D, int splits,
                                    cudaStream_t s);
cudaError_t launch_attn_merge(const AttnSplitParams& p, int D, cudaStream_t s);
cudaError_t configure_attn_split_kernels();

struct KvAppendParams {
    int B, L, Hkv, D, ctx_cap;
    const __nv_bfloat16* k_blk;  // [B][L][Hkv][D]
    const __nv_bfloat16* v_blk;
    __nv_bfloat16* k_ctx;        // [B][Hkv][ctx_cap][D]
    __nv_bfloat16* v_ctx;
    int32_t* ctx_len;            // [B], advanced by L where the block fits
    unsigned* status;
};

// Copies the block's K/V rows to cache positions ctx_len[b] .. ctx_len[b] + L - 1,
// then advances ctx_len[b] by L (two launches on stream s).
cudaError_t launch_kv_append(const KvAppendParams& p, cudaStream_t s);

struct CommitParams {
    const float* logits;
    int B, L, V, k;
    // Threshold mode (steps_left >= 1): a block commits its masked rows with
    // key <= kthr (confidence above gamma) and at least ceil(n / steps_left) of
    // its n masked rows; k is unused. steps_left == 0: a fixed budget of k.
    int steps_left;
    unsigned long long kthr;
    int slice;  // logits per CTA of a row's cluster (multiple of 4)
    const uint8_t* masked;
    int32_t* tok;
    uint8_t* masked_out;
    unsigned long long* key;  // [B*L]
    int32_t* arg;             // [B*L]
    // [2 + B], zero between calls: [0] clusters past their start-up mask
    // scan, [1] clusters finished, [2 + b] block b's ticket.
    unsigned* counters;
    int alias;  // masked_out is the masked buffer: no mask write before every scan is done
    unsigned* status;
    unsigned long long timeout_ns;
};

constexpr int kCommitCluster = 4;       // CTAs sharing one logit row
constexpr int kCommitSliceMax = 32768;  // fp32 logits per CTA (a quarter row at V = 131072)
constexpr int kCommitMaxL = 16384;      // rows per block

size_t commit_smem_bytes(int V, int L);
cudaError_t launch_commit(const CommitParams& p, cudaStream_t s);
int commit_max_clusters();  // co-resident clusters of the commit kernel (current device)
cudaError_t configure_commit_kernels();
cudaError_t configure_attn_kernels();

// LM head: logits[M][V] = hidden[M][K] * W[V][K]^T (bf16 in, fp32 out) on the
// tensor core; each row's maximum and first argmax go to rowmax (atomic max of
// key::enc_argmax, zero before the call).
struct LmHeadParams {
    int M, K, V;
    float* logits;
    unsigned long long* rowmax;  // [M]
    unsigned* status;
    unsigned long long timeout_ns;
};

// The commit step given each row's maximum / prediction (rowmax) — the
// fixed-budget or threshold rule as in CommitParams; key accumulates each
// row's fixed-point terms (zero before the call, zero after), blk counts each
// block's finished (row, chunk) units (zero before and after).
struct RowmaxCommitParams {
    const float* logits;
    int B, L, V, k, steps_left;
    unsigned long long kthr;
    const uint8_t* masked;
    int32_t* tok;
    uint8_t* masked_out;
    unsigned long long* key;     // [B*L] accumulators
    unsigned long long* rowmax;  // [B*L] from the LM head; zeroed per completed block
    unsigned* blk;               // [B]
    int32_t* arg;                // [B*L] predictions (out)
    unsigned long long* key_out; // [B*L] keys (out)
    unsigned* status;
    unsigned long long timeout_ns;
};

size_t lm_head_smem_bytes();
cudaError_t configure_lm_head_kernels();
cudaError_t launch_lm_head(const CUtensorMap& a, const CUtensorMap& b, const LmHeadParams& p, int num_sms,
                           cudaStream_t s);
cudaError_t launch_commit_rowmax(const RowmaxCommitParams& p, int num_sms, cudaStream_t s);

// Records "<where>: <msg>" as the calling thread's last host error (tt_last_error).
void record_host_error(const char* where, const char* msg);

}  // namespace tt
