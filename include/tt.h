/*
 * tt.h -- C ABI of the TwoTower denoising-step hot path on NVIDIA B300
 * (sm_103a): the denoiser's block attention and the unmask/commit step.
 *
 * Source of the method: "Nemotron-Labs-TwoTower: Diffusion Language Modeling
 * with Pretrained Autoregressive Context" (arXiv 2606.26493), Section 2.1
 * (two-tower architecture, "Bidirectional Attention", Eq. 1) and Section 2.2
 * ("Sampling", Algorithm 2, confidence unmasking).
 *
 * Conventions (all entry points):
 *   - Plain C types only. Tensor arguments are DEVICE pointers to contiguous
 *     row-major arrays with the shapes given below; the caller owns them.
 *   - The handle owns the scratch the kernels need (attention partials, the
 *     commit step's keys and predictions, and counters that every kernel
 *     leaves at zero). tt_create sizes it for the usual shapes; a call with a
 *     larger shape grows it first, which synchronizes the device and
 *     allocates. tt_reserve does that growth up front (e.g. before capturing a
 *     CUDA graph), after which no call of that size or smaller allocates.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls are asynchronous on it. Calls on one handle share its
 *     scratch, so their GPU work must be ordered (one stream, or events); use
 *     one handle per stream for concurrent work.
 *   - Return value: TT_OK, or a negative tt_status for an error detected on
 *     the host before anything is launched (nothing is written then). The
 *     message of the last host error of the calling thread is available from
 *     tt_last_error().
 *   - Errors detected on the device (a ctx_len outside [0, ctx_cap], a
 *     pipeline wait that timed out) set bits of the handle's status word; read
 *     and clear it with tt_get_error. Kernels never trap.
 *   - A handle may be used from one host thread at a time.
 */
#ifndef TT_H_
#define TT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TT_OK = 0,
    TT_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer             */
    TT_ERR_UNSUPPORTED = -2,  /* a shape outside the supported set (see below)          */
    TT_ERR_CUDA = -3,         /* a CUDA runtime or driver call failed                   */
    TT_ERR_TIMEOUT = -4,      /* tt_get_error: a bounded wait in a kernel gave up       */
    TT_ERR_DEVICE_CHECK = -5, /* tt_get_error: a kernel's argument check failed (ctx_len) */
    TT_ERR_NOT_READY = -6     /* tt_sync: the stream's work had not finished in time    */
} tt_status;

/* Bits of the device status word (tt_get_error). */
#define TT_DEV_CTX_LEN_RANGE 1 /* a ctx_len[b] outside [0, ctx_cap] (it was clamped), or a block
                                  that does not fit the cache (tt_kv_append skipped it) */
#define TT_DEV_WAIT_TIMEOUT 2  /* a bounded pipeline wait gave up; outputs invalid      */

typedef struct tt_context* tt_handle;

/* Shapes of one block-attention call (see the block attention section). */
typedef struct tt_attn_desc_s {
    int B, L, Hq, Hkv, D, ctx_cap;
    float scale; /* softmax scale; 0 selects 1/sqrt(D) */
} tt_attn_desc;

/* Creates a handle bound to CUDA device `device` (made current while the
 * library works on it). Allocates the device status word and the scratch for
 * the usual shapes (about 40 MB), and sets kernel attributes. Returns TT_OK,
 * TT_ERR_INVALID_ARG (handle NULL) or TT_ERR_CUDA (no such device, it is not
 * a compute capability 10.3 part, or an allocation failed). */
int tt_create(tt_handle* handle, int device);

/* Frees the handle and its scratch. Synchronizes nothing: the caller makes
 * sure no launch on the handle is still running. NULL is a no-op. */
int tt_destroy(tt_handle handle);

/* Grows the handle's scratch so that tt_block_attn / tt_block_attn_causal /
 * tt_kv_append with descriptor `attn` (may be NULL) and tt_commit /
 * tt_commit_threshold with B = commit_B, L = commit_L (0 for none) allocate
 * nothing when called. Synchronizes the device if it allocates. */
int tt_reserve(tt_handle handle, const tt_attn_desc* attn, int commit_B, int commit_L);

/* Reads and clears the device status word. Synchronizes the handle's device
 * (cudaDeviceSynchronize). *device_status receives the TT_DEV_* bits (may be
 * NULL). After a timeout it also zeroes the handle's counters (a call that
 * gave up may have left tickets behind). Returns TT_OK if no bit was set,
 * TT_ERR_TIMEOUT if a wait timed out, TT_ERR_DEVICE_CHECK if only an argument
 * check failed, TT_ERR_CUDA if the synchronization reported a CUDA error. */
int tt_get_error(tt_handle handle, int* device_status);

/* Waits on the host, for at most timeout_ms milliseconds, until the work
 * issued so far on `stream` (a cudaStream_t as void*, NULL = legacy default
 * stream) has finished, polling cudaStreamQuery; neither the device nor other
 * streams are synchronized, and nothing is cancelled. Returns TT_OK once the
 * stream has drained, with *device_status (may be NULL) = the TT_DEV_* bits of
 * the handle's status word, read but not cleared (tt_get_error clears them);
 * TT_ERR_NOT_READY if the work is still running after timeout_ms (it runs on:
 * call again, or tt_get_error); TT_ERR_CUDA if the stream reported an error.
 * timeout_ms = 0 looks once. A host-side watchdog for a serving loop: a call
 * whose kernels gave up a pipeline wait finishes within the handle's wait
 * limit (tt_set_wait_timeout) and shows TT_DEV_WAIT_TIMEOUT here. */
int tt_sync(tt_handle handle, void* stream, unsigned timeout_ms, int* device_status);

/* Sets how long a pipeline wait inside a kernel may last before it gives up,
 * sets TT_DEV_WAIT_TIMEOUT and lets the kernel wind down (default 1 s). */
int tt_set_wait_timeout(tt_handle handle, unsigned long long nanoseconds);

/* Tuning of the attention schedule (all attention entry points; results
 * agree within the attention tolerance whatever the schedule).
 *   kernel: 0 = chosen by shape (the default): the persistent schedule for
 *           caches of 16384 positions or more outside the training layout,
 *           one unit per CTA otherwise; 1 = one unit per CTA; 2 = persistent.
 *   max_ctas, min_tiles (persistent schedule): at most max_ctas CTAs (0 = one
 *           per SM) and at least min_tiles KV tiles of 128 keys per group of
 *           CTAs (0 = the default, 8; 1 cuts at any tile).
 *   splits (one-unit-per-CTA schedule): KV splits per unit (0 = by shape).
 * A unit is (sequence, KV head, pair of 128-row query tiles). */
int tt_set_attn_schedule(tt_handle handle, int kernel, int max_ctas, int min_tiles, int splits);

/* Kernel launches a tt_block_attn / tt_block_attn_causal call with this
 * descriptor makes on this handle under its current schedule (1, or 2 when a
 * unit is split and merged by a second kernel); a negative tt_status for an
 * invalid descriptor. */
int tt_block_attn_launches(tt_handle handle, const tt_attn_desc* desc);

/* Human-readable name of a tt_status value. */
const char* tt_status_string(int status);

/* Message of the last host-side error raised on the calling thread ("" if none). */
const char* tt_last_error(void);

/* ------------------------------------------------------------------------
 * Block attention -- Section 2.1, "Bidirectional Attention", Eq. (1):
 *   Attn(Q_b^(i), [K_<b^ctx,(i); K_b^den,(i)], [V_<b^ctx,(i); V_b^den,(i)])
 * Every query of the L-token noisy block takes ONE softmax over the
 * concatenation of the context tower's layer-i keys for the ctx_len[b] clean
 * positions before the block and the denoiser's own layer-i keys for the block,
 * with no mask inside the block. Layer alignment (denoiser layer i reads
 * context layer i) is the caller's choice of k_ctx / v_ctx: one call per layer.
 * GQA: query head h uses KV head h / (Hq / Hkv).
 *
 * Layouts (bf16, row-major, contiguous, 16-byte aligned):
 *   q      [B][L][Hq][D]        queries of the noisy block
 *   k_blk  [B][L][Hkv][D]       the block's own keys      (denoiser tower)
 *   v_blk  [B][L][Hkv][D]       the block's own values
 *   k_ctx  [B][Hkv][ctx_cap][D] layer-i KV cache           (context tower)
 *   v_ctx  [B][Hkv][ctx_cap][D]   positions >= ctx_len[b] are never used and
 *                                 may hold anything, NaN included
 *   ctx_len [B] int32, device    0 <= ctx_len[b] <= ctx_cap
 *   out    [B][L][Hq][D]        bf16, written in full
 * Arithmetic: bf16 products with fp32 accumulation (tcgen05), fp32 online
 * softmax, probabilities rounded to bf16 for the P*V product, output rounded
 * to bf16 (nearest even).
 * Supported: D in {64, 128}; Hq % Hkv == 0 with Hq/Hkv a power of two <= 128;
 * 1 <= L <= 65536; B >= 0 (B == 0 is a no-op); scale > 0 or 0 for 1/sqrt(D).
 * ------------------------------------------------------------------------ */
int tt_block_attn(tt_handle handle, const tt_attn_desc* desc, const void* q, const void* k_blk,
                  const void* v_blk, const void* k_ctx, const void* v_ctx,
                  const int32_t* ctx_len, void* out, void* stream);

/* ------------------------------------------------------------------------
 * Context-tower update after a commit -- Section 2.1, Algorithm 1: once a
 * block is clean, the context tower runs its
 * tokens causally over the prefix cache and the block's keys/values join the
 * cache. Per attention layer that is tt_block_attn_causal followed by
 * tt_kv_append.
 *
 * tt_block_attn_causal: the same call as tt_block_attn (same arguments,
 * layouts, arithmetic and errors) except that block query l sees
 * the ctx_len[b] cache positions and block keys 0..l only:
 *   out[b][l][h] = softmax over [K_ctx[0..C_b-1]; K_blk[0..l]] applied to V.
 * With L == 1 it equals tt_block_attn (one autoregressive decode row).
 * ------------------------------------------------------------------------ */
int tt_block_attn_causal(tt_handle handle, const tt_attn_desc* desc, const void* q,
                         const void* k_blk, const void* v_blk, const void* k_ctx,
                         const void* v_ctx, const int32_t* ctx_len, void* out, void* stream);

/* tt_kv_append: copies the block's keys and values into the cache behind the
 * positions already there and advances the lengths:
 *   k_ctx[b][h][ctx_len[b] + l][:] = k_blk[b][l][h][:]   (same for v), l < L
 *   ctx_len[b] += L
 * for every b with 0 <= ctx_len[b] <= ctx_cap - L. A block that does not fit
 * is skipped (cache and ctx_len[b] unchanged) and sets TT_DEV_CTX_LEN_RANGE.
 * desc gives B, L, Hkv, D and ctx_cap (Hq and scale are not used);
 * layouts as for tt_block_attn: k_blk/v_blk [B][L][Hkv][D] bf16, k_ctx/v_ctx
 * [B][Hkv][ctx_cap][D] bf16 (written), ctx_len [B] int32 (read and written),
 * all device pointers, 16-byte aligned. Cache rows outside the appended range
 * are not touched. Two launches on `stream` (the copy, then the lengths), no
 * scratch. Supported: D in {64, 128}, 1 <= L <= ctx_cap, Hkv >= 1, B >= 0.
 * Host errors: TT_ERR_INVALID_ARG for a NULL or misaligned pointer or a
 * descriptor outside the supported range.
 * ------------------------------------------------------------------------ */
int tt_kv_append(tt_handle handle, const tt_attn_desc* desc, const void* k_blk, const void* v_blk,
                 void* k_ctx, void* v_ctx, int32_t* ctx_len, void* stream);

/* ------------------------------------------------------------------------
 * Training-time batched block attention -- Section 2.3, "Implementation":
 * the denoiser processes all noisy blocks of a clean sequence in one forward
 * pass; its attention attends to the past clean blocks (the frozen context
 * tower's keys/values of the clean sequence) and bidirectionally within the
 * current noisy block. For a sequence of N = n*S tokens, noisy block j
 * (tokens j*S .. j*S+S-1) takes, per query, one softmax over
 *   [K_clean[0 .. j*S-1] ; K_noisy[j*S .. j*S+S-1]]   (block 0: its own keys only)
 * applied to the matching values. This is tt_block_attn over the B*n noisy
 * blocks with ctx_len = j*S, every block of a sequence reading that
 * sequence's clean cache; arithmetic, tolerance and errors as there.
 *
 * Layouts (bf16, row-major, contiguous, 16-byte aligned, device):
 *   q        [B][N][Hq][D]    queries of the noisy tokens
 *   k_noisy  [B][N][Hkv][D]   keys/values of the noisy tokens (denoiser)
 *   v_noisy  [B][N][Hkv][D]
 *   k_clean  [B][Hkv][N][D]   keys/values of the clean tokens (context tower)
 *   v_clean  [B][Hkv][N][D]     only positions below the block's start are read
 *   out      [B][N][Hq][D]
 * Supported: as tt_block_attn with L = S; N a multiple of S; B*N/S <= 65535.
 * ------------------------------------------------------------------------ */
typedef struct {
    int B, N, S, Hq, Hkv, D;
    float scale; /* softmax scale; 0 selects 1/sqrt(D) */
} tt_train_desc;

int tt_block_attn_train(tt_handle handle, const tt_train_desc* desc, const void* q,
                        const void* k_noisy, const void* v_noisy, const void* k_clean,
                        const void* v_clean, void* out, void* stream);

/* ------------------------------------------------------------------------
 * Unmask / commit -- Section 2.2, "Sampling", Algorithm 2 (ConfidenceSample),
 * read as a fixed budget of k commits per block per step (the threshold rule
 * with gamma > 1 and T = L/k steps).
 * For every row r of block b with masked[r] == 1:
 *   prediction a_r = lowest v with logits[r][v] == max_v logits[r][v]
 *   key_r = sum_v rint(2^40 * e(RN32(logits[r][v] - max))), an integer;
 *     e is an fp32 exponential fixed by this library (Cody-Waite reduction,
 *     degree-7 Taylor polynomial, fused multiply-adds; within 1 ulp of exp
 *     on [-30, 0], 0 below -30), so the key is bit-reproducible;
 *     2^40 / key_r is the maximum softmax probability (the confidence) up to
 *     a relative error below V * 2^-40 + 2^-22.
 * Then per block the min(k, #masked) rows with the smallest (key, row) are
 * committed: tok[r] = a_r, masked_out[r] = 0. Every other entry of tok is left
 * untouched; masked_out[r] = masked[r] elsewhere.
 *
 *   logits     [B*L][V] fp32, device, 16-byte aligned, finite values
 *   masked     [B*L] uint8 (0/1), device
 *   tok        [B*L] int32, device, updated in place at committed rows
 *   masked_out [B*L] uint8, device; may be the same buffer as masked
 * Rows with masked[r] == 0 are not read. Supported: V % 4 == 0,
 * 4 <= V <= 131072, 1 <= L <= 16384, k >= 1 (k >= #masked commits all).
 * masked and masked_out are the same buffer or do not overlap
 * (TT_ERR_INVALID_ARG otherwise). The key and prediction of every row that was
 * masked on entry stay in the handle's scratch until the next call on the
 * handle (tt_commit_keys copies them out).
 * ------------------------------------------------------------------------ */
int tt_commit(tt_handle handle, const float* logits, int B, int L, int V, const uint8_t* masked,
              int k, int32_t* tok, uint8_t* masked_out, void* stream);

/* Copies the keys (uint64 [rows]) and predictions (int32 [rows]) that the last
 * tt_commit / tt_commit_threshold call on this handle computed into device
 * buffers key_dst / arg_dst (either may be NULL), asynchronously on `stream`.
 * Entries of rows that were not masked in that call are unspecified. rows =
 * B*L of that call. A debugging and testing aid (the canonical keys are what
 * the committed set is decided on). */
int tt_commit_keys(tt_handle handle, uint64_t* key_dst, int32_t* arg_dst, int rows, void* stream);

/* ------------------------------------------------------------------------
 * Unmask / commit with a confidence threshold -- Section 2.2, Algorithm 2,
 * ConfidenceSample read as: at denoising step r of T, a block commits every
 * still-masked position whose confidence exceeds gamma, and never fewer than
 * ceil(#masked / (T - r + 1)) of its most confident masked positions, so that
 * the block is complete after T steps (steps_left = T - r + 1; with
 * steps_left = 1 every masked position commits).
 * The confidence of row r is 2^40 / key_r (key and prediction as in
 * tt_commit); "confidence > gamma" is decided exactly as gamma * key_r < 2^40
 * in integer arithmetic (gamma as the double given). The rows that pass are
 * the first ones of the (key, row) order, so the committed set is the first
 * max(#passing, ceil(#masked / steps_left)) masked rows of each block in that
 * order. gamma <= 0 commits every masked row; gamma >= 1 reduces to the floor.
 * Arguments, layouts, scratch and errors as tt_commit; gamma must not be NaN
 * and steps_left must be >= 1.
 * ------------------------------------------------------------------------ */
int tt_commit_threshold(tt_handle handle, const float* logits, int B, int L, int V,
                        const uint8_t* masked, double gamma, int steps_left, int32_t* tok,
                        uint8_t* masked_out, void* stream);

/* ------------------------------------------------------------------------
 * The denoiser's LM head with the commit step behind it -- Section 2.2,
 * Algorithm 2: the denoiser's distribution over the vocabulary for every
 * position of the block, then ConfidenceSample on it.
 *
 * tt_lm_head: logits[m][v] = sum_k hidden[m][k] * weight[v][k], bf16 inputs,
 * fp32 accumulation on the tensor core, fp32 logits out (written in full).
 * Its epilogue also finds each row's maximum and first argmax and leaves
 * them in the handle for the next tt_commit_rowmax call on the handle (a new
 * tt_lm_head replaces them).
 *   hidden [M][K] bf16, weight [V][K] bf16, logits [M][V] fp32; device
 *   pointers, 16-byte aligned; K % 8 == 0, V % 4 == 0, K >= 8, V >= 4.
 * Two launches (the row maxima are cleared first).
 *
 * tt_commit_rowmax: the same step as tt_commit (same rule, keys, tie-breaks,
 * results, in-place masks allowed) on the logits of the last tt_lm_head call
 * (B*L == its M, V == its V; TT_ERR_INVALID_ARG otherwise), using the row
 * maxima and predictions it found instead of a pass of its own. One launch.
 * The commit is bit-identical to tt_commit on the same logits.
 * ------------------------------------------------------------------------ */
int tt_lm_head(tt_handle handle, const void* hidden, const void* weight, int M, int K, int V,
               float* logits, void* stream);

int tt_commit_rowmax(tt_handle handle, const float* logits, int B, int L, int V,
                     const uint8_t* masked, int k, int32_t* tok, uint8_t* masked_out, void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free commit. The paper has no counterpart of this entry point:
 * it is the same step as tt_commit, for callers that cannot allocate device
 * memory -- a serving engine that reserves all of HBM for its own pool at
 * start-up, or a plug-in host that forbids allocation while a request runs --
 * and so can neither call cudaMalloc nor create a handle (whose scratch is
 * allocated).
 *
 * Arguments and results are those of tt_commit without the handle; the
 * scratch (per-row keys and predictions, per-block tickets, a status word)
 * is a fixed array of about 1 MiB built into the library, present on every
 * GPU that loads it until the process exits. Limits: B*L <= 65536 (larger
 * sizes return TT_ERR_UNSUPPORTED with a message in tt_last_error), plus
 * those of tt_commit. Works on the current CUDA device. The first call on a
 * device sets that device up (looks up the array's device address, sets
 * kernel attributes); with CUDA's lazy module loading that first call may
 * also load the library's device code and so allocate, so make it (or a
 * warm-up call) at start-up and before any stream capture. Later calls clear
 * the tickets on `stream` (cudaMemsetAsync) and allocate nothing.
 * All calls share the one array: calls whose GPU work overlaps (other
 * streams, other threads) race and must be ordered by the caller.
 * ------------------------------------------------------------------------ */
int tt_commit_noalloc(const float* logits, int B, int L, int V, const uint8_t* masked, int k,
                      int32_t* tok, uint8_t* masked_out, void* stream);

/* Reads and clears the status word of tt_commit_noalloc's built-in scratch on
 * the current device (TT_DEV_* bits: a wait that timed out makes that call's
 * outputs invalid). Synchronizes the device. Returns TT_OK, TT_ERR_TIMEOUT
 * (the timeout bit was set; the tickets are cleared by the next call anyway)
 * or TT_ERR_CUDA. The device must have made a tt_commit_noalloc call. */
int tt_commit_noalloc_status(int* device_status);

#ifdef __cplusplus
}
#endif

#endif /* TT_H_ */
