// C-ABI layer: argument checks, launch planning (KV splits), TMA tensor-map
// encoding and kernel launches. See include/tt.h for the contract.
#include <cudaTypedefs.h>

#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>

#include "host_trace.h"
#include "tt.h"
#include "tt_internal.h"

struct tt_context {
    int device;
    int num_sms;
    unsigned* status;  // device word, TT_DEV_* bits
    unsigned long long timeout_ns;
    // Workspace owned by the handle: attention partials or commit keys and
    // predictions (calls on one handle are ordered on the GPU, so they share
    // it), and counters that every kernel leaves at zero.
    void* ws;
    size_t ws_bytes;
    unsigned* ctr;
    size_t ctr_count;
    int attn_kernel;  // attention schedule: 0 by shape, 1 one unit per CTA, 2 persistent
    int max_ctas;     // persistent schedule: CTAs at most (0: one per SM)
    int min_tiles;    // persistent schedule: KV tiles per group at least
    int splits;       // one-unit-per-CTA schedule: KV splits per unit (0: by shape)
    // Encoded TMA descriptors of recent calls (encoding one costs microseconds
    // of host time; a caller that reuses its buffers hits this cache).
    struct MapEntry {
        void* base;
        int rank;
        cuuint64_t dims[5], strides[4];
        cuuint32_t box[5];
        unsigned long long used;
        CUtensorMap map;
    };
    MapEntry maps[32];
    unsigned long long map_clock;
    // LM head -> commit hand-off: per-row maxima and key accumulators [rows]
    // (u64 each) and block tickets [blocks] (u32), zero between calls; the
    // shape of the last tt_lm_head call.
    void* lm;
    size_t lm_rows, lm_blocks;
    int lm_M, lm_V;
};

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Makes the handle's device current for the scope of a call.
class DeviceGuard {
public:
    explicit DeviceGuard(int dev) {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess;
        if (ok_ && prev_ != dev) ok_ = cudaSetDevice(dev) == cudaSuccess;
        else if (ok_) prev_ = -1;
    }
    ~DeviceGuard() {
        if (ok_ && prev_ >= 0) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

private:
    int prev_ = -1;
    bool ok_ = false;
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }


struct AttnPlan {
    int G, n_mtiles, n_pairs, nblk, width, ngroups;
    size_t part_o_bytes, ws_bytes, ctr_count;
};

// Largest divisor of n that is <= cap.
int divisor_at_most(int n, int cap) {
    for (int w = cap < n ? cap : n; w > 1; --w)
        if (n % w == 0) return w;
    return 1;
}

// Checks a descriptor; fills the launch plan. `cache_seqs` = sequences of the
// context cache (B, or fewer in the training layout). Schedule: one CTA per SM
// (at most max_ctas), in groups of `width` CTAs that take the pairs of a pair
// block together. The width is a divisor of the pair count: up to 4 when the
// whole cache fits comfortably in L2 (any order then reads it once from HBM),
// up to 16 otherwise, so that the pairs reading one K/V tile run at the same
// time.
int plan_attn(const tt_attn_desc* d, int num_sms, int max_ctas, int cache_seqs, AttnPlan* pl) {
    if (!d) return fail(TT_ERR_INVALID_ARG, "tt_block_attn: desc is NULL");
    if (d->B < 0 || d->B > 65535) return fail(TT_ERR_INVALID_ARG, "B=%d outside [0, 65535]", d->B);
    if (d->L < 1 || d->L > 65536) return fail(TT_ERR_INVALID_ARG, "L=%d outside [1, 65536]", d->L);
    if (d->Hq < 1 || d->Hkv < 1 || d->Hkv > 65535 || d->Hq % d->Hkv)
        return fail(TT_ERR_INVALID_ARG, "Hq=%d must be a positive multiple of Hkv=%d", d->Hq, d->Hkv);
    const int G = d->Hq / d->Hkv;
    if (G > 128 || (G & (G - 1)))
        return fail(TT_ERR_UNSUPPORTED, "Hq/Hkv=%d must be a power of two <= 128", G);
    if (d->D != 64 && d->D != 128)
        return fail(TT_ERR_UNSUPPORTED, "head dim D=%d unsupported (64 or 128)", d->D);
    if (d->ctx_cap < 0 || d->ctx_cap > (1 << 24))
        return fail(TT_ERR_INVALID_ARG, "ctx_cap=%d outside [0, 2^24]", d->ctx_cap);
    if (!(d->scale >= 0.f) || std::isinf(d->scale))
        return fail(TT_ERR_INVALID_ARG, "scale must be finite and >= 0");
    pl->G = G;
    pl->n_mtiles = static_cast<int>((static_cast<long>(G) * d->L + tt::kTile - 1) / tt::kTile);
    pl->n_pairs = (pl->n_mtiles + 1) / 2;
    pl->nblk = (d->L + tt::kTile - 1) / tt::kTile;
    const double kv_bytes = 4.0 * cache_seqs * d->Hkv * static_cast<double>(d->ctx_cap) * d->D;
    pl->width = divisor_at_most(pl->n_pairs, kv_bytes > 48e6 ? 16 : 4);
    int ctas = num_sms;
    if (max_ctas > 0 && max_ctas < ctas) ctas = max_ctas;
    pl->ngroups = ctas / pl->width > 0 ? ctas / pl->width : 1;
    const size_t slots = 2 * static_cast<size_t>(pl->ngroups) * pl->width;
    pl->part_o_bytes = align256(slots * tt::attn_slot_o_floats(d->D) * sizeof(float));
    pl->ws_bytes = pl->part_o_bytes + align256(slots * tt::attn_slot_ml(d->D) * sizeof(float2));
    pl->ctr_count = static_cast<size_t>(d->B) * d->Hkv * pl->n_mtiles;
    return TT_OK;
}

// The one-unit-per-CTA schedule's KV split: the split count minimising
// waves * (tiles per split + 2) over the capacity's tiles (one CTA per SM; the
// +2 stands for a CTA's prologue and epilogue; a split also pays for the
// merge), or `forced` splits. Fills splits, chunk and the partials' bytes.
struct SplitPlan {
    int splits, chunk;
    size_t ws_o_bytes, ws_bytes;
};

SplitPlan plan_split(const tt_attn_desc* d, const AttnPlan& pl, int num_sms, int forced) {
    SplitPlan sp;
    const int nt_max = (d->ctx_cap + tt::kTile - 1) / tt::kTile + pl.nblk;
    const long units = static_cast<long>(d->B) * d->Hkv * pl.n_pairs;
    int best = 1;
    if (forced > 0) {
        best = forced < nt_max ? forced : nt_max;
    } else if (units > 0) {
        double best_cost = 1e300;
        const int smax = nt_max < 64 ? nt_max : 64;
        for (int s = 1; s <= smax; ++s) {
            const int chunk = (nt_max + s - 1) / s;
            const int s2 = (nt_max + chunk - 1) / chunk;
            if (s2 != s) continue;
            const long waves = (units * s2 + num_sms - 1) / num_sms;
            const double cost = static_cast<double>(waves) * (chunk + 2) + (s2 > 1 ? 2 : 0);
            if (cost < best_cost) { best_cost = cost; best = s2; }
        }
    }
    sp.chunk = (nt_max + best - 1) / best;
    sp.splits = (nt_max + sp.chunk - 1) / sp.chunk;
    if (sp.splits > 1) {
        const size_t rows = static_cast<size_t>(sp.splits) * d->B * d->Hkv *
                            static_cast<size_t>(pl.n_mtiles) * tt::kTile;
        sp.ws_o_bytes = align256(rows * d->D * sizeof(float));
        sp.ws_bytes = sp.ws_o_bytes + align256(rows * 2 * sizeof(float));
    } else {
        sp.ws_o_bytes = sp.ws_bytes = 0;
    }
    return sp;
}

// Which attention schedule a call takes: the persistent stream-K kernel for
// long caches (its per-range cost is small against long units, and it
// balances ragged lengths), one unit per CTA otherwise (faster per tile on
// short or equal-length units, and for the training layout's many short
// units).
bool use_persistent(const tt_context* h, const tt_attn_desc* d, int ctx_group) {
    if (h->attn_kernel == 1) return false;
    if (h->attn_kernel == 2) return true;
    return !ctx_group && d->ctx_cap >= 16384;
}

size_t commit_ws_bytes(size_t rows) { return align256(rows * 8) + align256(rows * 4); }

// Grows the handle's workspace and counters to at least the given sizes. A
// growth synchronizes the device (the old buffers may still be in use) and
// allocates; the new counters are zeroed.
int ensure_workspace(tt_context* h, size_t ws_bytes, size_t ctr_count) {
    cudaError_t e;
    if (ws_bytes > h->ws_bytes) {
        const size_t n = (ws_bytes + (1u << 20) - 1) & ~static_cast<size_t>((1u << 20) - 1);
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        if (h->ws) cudaFree(h->ws);
        h->ws = nullptr;
        h->ws_bytes = 0;
        if ((e = cudaMalloc(&h->ws, n)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
        h->ws_bytes = n;
    }
    if (ctr_count > h->ctr_count) {
        const size_t n = (ctr_count + 4095) & ~static_cast<size_t>(4095);
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        if (h->ctr) cudaFree(h->ctr);
        h->ctr = nullptr;
        h->ctr_count = 0;
        if ((e = cudaMalloc(&h->ctr, n * sizeof(unsigned))) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(counters)");
        if ((e = cudaMemset(h->ctr, 0, n * sizeof(unsigned))) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(counters)");
        h->ctr_count = n;
    }
    return TT_OK;
}

int encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box, const char* name);

// encode() through the handle's descriptor cache (least recently used out).
int encode_cached(tt_context* h, CUtensorMap* m, void* base, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, const char* name) {
    tt_context::MapEntry* victim = &h->maps[0];
    for (auto& e : h->maps) {
        if (e.used && e.base == base && e.rank == rank &&
            !std::memcmp(e.dims, dims, sizeof(cuuint64_t) * rank) &&
            !std::memcmp(e.strides, strides, sizeof(cuuint64_t) * (rank - 1)) &&
            !std::memcmp(e.box, box, sizeof(cuuint32_t) * rank)) {
            e.used = ++h->map_clock;
            *m = e.map;
            return TT_OK;
        }
        if (e.used < victim->used) victim = &e;
    }
    const int st = encode(m, base, rank, dims, strides, box, name);
    if (st != TT_OK) return st;
    victim->base = base;
    victim->rank = rank;
    std::memcpy(victim->dims, dims, sizeof(cuuint64_t) * rank);
    std::memcpy(victim->strides, strides, sizeof(cuuint64_t) * (rank - 1));
    std::memcpy(victim->box, box, sizeof(cuuint32_t) * rank);
    victim->map = *m;
    victim->used = ++h->map_clock;
    return TT_OK;
}

int encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box, const char* name) {
    auto fn = encode_fn();
    if (!fn) return fail(TT_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (driver too old?)");
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(TT_ERR_CUDA, "tensor map for %s: CUresult %d", name, (int)r);
    return TT_OK;
}

// Checks a training-layout descriptor and gives the equivalent per-block one.
int train_desc(const tt_train_desc* t, tt_attn_desc* d) {
    if (!t) return fail(TT_ERR_INVALID_ARG, "tt_block_attn_train: desc is NULL");
    if (t->B < 0) return fail(TT_ERR_INVALID_ARG, "B=%d < 0", t->B);
    if (t->S < 1 || t->N < t->S || t->N % t->S)
        return fail(TT_ERR_INVALID_ARG, "N=%d must be a positive multiple of the block size S=%d",
                    t->N, t->S);
    const long blocks = static_cast<long>(t->B) * (t->N / t->S);
    if (blocks > 65535)
        return fail(TT_ERR_UNSUPPORTED, "B * N / S = %ld noisy blocks (at most 65535)", blocks);
    d->B = static_cast<int>(blocks);
    d->L = t->S;
    d->Hq = t->Hq;
    d->Hkv = t->Hkv;
    d->D = t->D;
    d->ctx_cap = t->N;
    d->scale = t->scale;
    return TT_OK;
}

}  // namespace

void tt::record_host_error(const char* where, const char* msg) { fail(0, "%s: %s", where, msg); }

extern "C" {

const char* tt_status_string(int s) {
    switch (s) {
        case TT_OK: return "TT_OK";
        case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG";
        case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED";
        case TT_ERR_CUDA: return "TT_ERR_CUDA";
        case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT";
        case TT_ERR_DEVICE_CHECK: return "TT_ERR_DEVICE_CHECK";
        case TT_ERR_NOT_READY: return "TT_ERR_NOT_READY";
        default: return "TT_ERR_UNKNOWN";
    }
}

const char* tt_last_error(void) { return g_last_error.c_str(); }

int tt_create(tt_handle* out, int device) {
    if (!out) return fail(TT_ERR_INVALID_ARG, "tt_create: handle pointer is NULL");
    *out = nullptr;
    int n = 0;
    cudaError_t e = cudaGetDeviceCount(&n);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= n) return fail(TT_ERR_CUDA, "device %d not present (%d devices)", device, n);
    DeviceGuard g(device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", device);
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, device)) != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
        return fail(TT_ERR_CUDA, "device %d is sm_%d%d; this library is built for sm_103a", device,
                    prop.major, prop.minor);
    if ((e = tt::configure_attn_kernels()) != cudaSuccess) return cuda_fail(e, "attention kernel attributes");
    if ((e = tt::configure_attn_split_kernels()) != cudaSuccess)
        return cuda_fail(e, "attention kernel attributes");
    if ((e = tt::configure_commit_kernels()) != cudaSuccess) return cuda_fail(e, "commit kernel attributes");
    if ((e = tt::configure_lm_head_kernels()) != cudaSuccess) return cuda_fail(e, "LM head kernel attributes");
    tt_context* h = new tt_context();
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    h->timeout_ns = 1000000000ull;
    h->min_tiles = 8;
    if ((e = cudaMalloc(&h->status, sizeof(unsigned))) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaMalloc(status)");
    }
    if ((e = cudaMemset(h->status, 0, sizeof(unsigned))) != cudaSuccess) {
        cudaFree(h->status);
        delete h;
        return cuda_fail(e, "cudaMemset(status)");
    }
    // The attention partials of a full grid at D = 128 and 64 Ki counters up
    // front, so that the usual shapes never allocate on the call path.
    const size_t slots = 2 * static_cast<size_t>(h->num_sms);
    const size_t ws0 = align256(slots * tt::attn_slot_o_floats(128) * sizeof(float)) +
                       align256(slots * tt::attn_slot_ml(128) * sizeof(float2));
    const int st = ensure_workspace(h, ws0, 65536);
    if (st != TT_OK) {
        tt_destroy(h);
        return st;
    }
    *out = h;
    return TT_OK;
}

int tt_destroy(tt_handle h) {
    if (!h) return TT_OK;
    DeviceGuard g(h->device);
    cudaFree(h->status);
    if (h->ws) cudaFree(h->ws);
    if (h->ctr) cudaFree(h->ctr);
    if (h->lm) cudaFree(h->lm);
    delete h;
    return TT_OK;
}

int tt_set_wait_timeout(tt_handle h, unsigned long long ns) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "handle is NULL");
    if (ns == 0) return fail(TT_ERR_INVALID_ARG, "timeout must be > 0");
    h->timeout_ns = ns;
    return TT_OK;
}

int tt_set_attn_schedule(tt_handle h, int kernel, int max_ctas, int min_tiles, int splits) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "handle is NULL");
    if (kernel < 0 || kernel > 2) return fail(TT_ERR_INVALID_ARG, "kernel must be 0, 1 or 2");
    if (max_ctas < 0 || min_tiles < 0 || splits < 0)
        return fail(TT_ERR_INVALID_ARG, "max_ctas, min_tiles and splits must be >= 0");
    h->attn_kernel = kernel;
    h->max_ctas = max_ctas;
    h->min_tiles = min_tiles > 0 ? min_tiles : 8;
    h->splits = splits;
    return TT_OK;
}

int tt_reserve(tt_handle h, const tt_attn_desc* attn, int commit_B, int commit_L) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_reserve: handle is NULL");
    if (commit_B < 0 || commit_L < 0) return fail(TT_ERR_INVALID_ARG, "tt_reserve: negative size");
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    size_t ws = 0, ctr = 0;
    if (attn) {
        AttnPlan pl;
        const int st = plan_attn(attn, h->num_sms, h->max_ctas, attn->B, &pl);
        if (st != TT_OK) return st;
        const SplitPlan sp = plan_split(attn, pl, h->num_sms, h->splits);
        ws = pl.ws_bytes > sp.ws_bytes ? pl.ws_bytes : sp.ws_bytes;
        ctr = pl.ctr_count;
    }
    const size_t rows = static_cast<size_t>(commit_B) * commit_L;
    if (commit_ws_bytes(rows) > ws) ws = commit_ws_bytes(rows);
    if (2 + static_cast<size_t>(commit_B) > ctr) ctr = 2 + static_cast<size_t>(commit_B);
    return ensure_workspace(h, ws, ctr);
}

int tt_block_attn_launches(tt_handle h, const tt_attn_desc* d) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_block_attn_launches: handle is NULL");
    AttnPlan pl;
    const int st = plan_attn(d, h->num_sms, h->max_ctas, d ? d->B : 0, &pl);
    if (st != TT_OK) return st;
    if (d->B == 0) return 0;
    if (use_persistent(h, d, 0)) return 1;
    return plan_split(d, pl, h->num_sms, h->splits).splits > 1 ? 2 : 1;
}

int tt_get_error(tt_handle h, int* device_status) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "handle is NULL");
    DeviceGuard g(h->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned v = 0;
    if ((e = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "read status");
    if ((e = cudaMemset(h->status, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "clear status");
    // A call that gave up on a wait may have left tickets behind.
    if ((v & TT_DEV_WAIT_TIMEOUT) && h->ctr &&
        (e = cudaMemset(h->ctr, 0, h->ctr_count * sizeof(unsigned))) != cudaSuccess)
        return cuda_fail(e, "clear counters");
    if ((v & TT_DEV_WAIT_TIMEOUT) && h->lm &&
        (e = cudaMemset(h->lm, 0, h->lm_rows * 16 + h->lm_blocks * 4)) != cudaSuccess)
        return cuda_fail(e, "clear counters");
    if (device_status) *device_status = static_cast<int>(v);
    if (v & TT_DEV_WAIT_TIMEOUT) return TT_ERR_TIMEOUT;
    return v ? TT_ERR_DEVICE_CHECK : TT_OK;
}

int tt_sync(tt_handle h, void* stream, unsigned timeout_ms, int* device_status) {
    if (device_status) *device_status = 0;
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_sync: handle is NULL");
    DeviceGuard g(h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaStreamQuery(s);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) return cuda_fail(e, "tt_sync: cudaStreamQuery");
        if (std::chrono::steady_clock::now() - t0 >= std::chrono::milliseconds(timeout_ms))
            return fail(TT_ERR_NOT_READY, "tt_sync: the stream is still busy after %u ms", timeout_ms);
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    // The stream has drained: this copy waits for nothing else on it.
    unsigned v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, h->status, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "tt_sync: read status");
    if (device_status) *device_status = static_cast<int>(v);
    return TT_OK;
}

}  // extern "C"

// Body of tt_block_attn (causal = 0), tt_block_attn_causal (causal = 1) and
// tt_block_attn_train (ctx_group = blocks per clean sequence: d->B counts the
// noisy blocks, the caches belong to d->B / ctx_group clean sequences and
// ctx_len is implied).
static int block_attn_call(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                           const void* v_blk, const void* k_ctx, const void* v_ctx,
                           const int32_t* ctx_len, void* out, void* stream, int causal,
                           int ctx_group = 0) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_block_attn: handle is NULL");
    AttnPlan pl;
    const int cache_seqs = d && ctx_group ? d->B / ctx_group : (d ? d->B : 0);
    int st = plan_attn(d, h->num_sms, h->max_ctas, cache_seqs, &pl);
    if (st != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!q || !k_blk || !v_blk || (!ctx_len && !ctx_group) || !out)
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: a tensor pointer is NULL");
    if (d->ctx_cap > 0 && (!k_ctx || !v_ctx))
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: k_ctx/v_ctx NULL with ctx_cap > 0");
    if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out) ||
        (d->ctx_cap > 0 && (!aligned16(k_ctx) || !aligned16(v_ctx))))
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: tensors must be 16-byte aligned");
    if (ctx_len && (reinterpret_cast<uintptr_t>(ctx_len) & 3u))
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: ctx_len must be 4-byte aligned");
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    const bool persistent = use_persistent(h, d, ctx_group);
    const SplitPlan sp = persistent ? SplitPlan{1, 0, 0, 0} : plan_split(d, pl, h->num_sms, h->splits);
    if ((st = ensure_workspace(h, persistent ? pl.ws_bytes : sp.ws_bytes, persistent ? pl.ctr_count : 0)) !=
        TT_OK)
        return st;

    const int B = d->B, L = d->L, Hq = d->Hq, Hkv = d->Hkv, D = d->D, G = pl.G;
    const cuuint64_t e2 = 2;  // bytes per bf16
    tt::AttnMaps maps;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)L,
                                    (cuuint64_t)B};
        const cuuint64_t str[4] = {D * e2, (cuuint64_t)G * D * e2, (cuuint64_t)Hq * D * e2,
                                   (cuuint64_t)L * Hq * D * e2};
        const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)(tt::kTile / G), 1};
        if ((st = encode_cached(h, &maps.q, const_cast<void*>(q), 5, dims, str, box, "q")) != TT_OK) return st;
    }
    {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)L, (cuuint64_t)B};
        const cuuint64_t str[3] = {D * e2, (cuuint64_t)Hkv * D * e2, (cuuint64_t)L * Hkv * D * e2};
        const cuuint32_t box[4] = {64, 1, (cuuint32_t)tt::kTile, 1};
        if ((st = encode_cached(h, &maps.k_blk, const_cast<void*>(k_blk), 4, dims, str, box, "k_blk")) != TT_OK)
            return st;
        if ((st = encode_cached(h, &maps.v_blk, const_cast<void*>(v_blk), 4, dims, str, box, "v_blk")) != TT_OK)
            return st;
    }
    {
        // With no cache (ctx_cap == 0) no context tile is ever loaded; the maps
        // only need to be well formed, so they point at the block keys.
        const bool none = d->ctx_cap == 0;
        const cuuint64_t dims[3] = {(cuuint64_t)D, none ? (cuuint64_t)tt::kTile : (cuuint64_t)d->ctx_cap,
                                    none ? 1 : (cuuint64_t)cache_seqs * Hkv};
        const cuuint64_t str[2] = {D * e2, (none ? (cuuint64_t)tt::kTile : (cuuint64_t)d->ctx_cap) * D * e2};
        const cuuint32_t box[3] = {64, (cuuint32_t)tt::kTile, 1};
        void* kc = none ? const_cast<void*>(k_blk) : const_cast<void*>(k_ctx);
        void* vc = none ? const_cast<void*>(v_blk) : const_cast<void*>(v_ctx);
        if ((st = encode_cached(h, &maps.k_ctx, kc, 3, dims, str, box, "k_ctx")) != TT_OK) return st;
        if ((st = encode_cached(h, &maps.v_ctx, vc, 3, dims, str, box, "v_ctx")) != TT_OK) return st;
    }
    const float scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(D));
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!persistent) {
        tt::AttnSplitParams q;
        q.B = B; q.L = L; q.Hq = Hq; q.Hkv = Hkv; q.G = G; q.ctx_cap = d->ctx_cap;
        q.n_mtiles = pl.n_mtiles; q.n_pairs = pl.n_pairs; q.nblk = pl.nblk;
        q.causal = causal;
        q.ctx_group = ctx_group;
        q.chunk = sp.chunk;
        q.scale_log2 = scale * 1.4426950408889634f;
        q.ctx_len = ctx_len;
        q.out = static_cast<__nv_bfloat16*>(out);
        q.ws_o = sp.splits > 1 ? static_cast<float*>(h->ws) : nullptr;
        q.ws_ml = sp.splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(h->ws) + sp.ws_o_bytes)
                                : nullptr;
        q.status = h->status;
        q.timeout_ns = h->timeout_ns;
        cudaError_t e = tt::launch_block_attn_split(maps, q, D, sp.splits, cs);
        if (e != cudaSuccess) return cuda_fail(e, "block attention launch");
        if (sp.splits > 1 && (e = tt::launch_attn_merge(q, D, cs)) != cudaSuccess)
            return cuda_fail(e, "split merge launch");
        return TT_OK;
    }
    tt::AttnParams p;
    p.B = B; p.L = L; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.ctx_cap = d->ctx_cap;
    p.n_mtiles = pl.n_mtiles; p.n_pairs = pl.n_pairs; p.nblk = pl.nblk;
    p.causal = causal;
    p.ctx_group = ctx_group;
    p.width = pl.width;
    p.ngroups = pl.ngroups;
    p.min_tiles = h->min_tiles;
    // Measured fixed costs, in KV tiles' time: a unit's (Q load, pipeline
    // start, epilogue) about 4 for short units; a cut's (partial out, ticket,
    // merge) about 8. Every range stays longer than a unit's fixed cost.
    p.item_cost = h->min_tiles > 4 ? 4 : h->min_tiles - 1;
    p.cut_cost = 8;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.ctx_len = ctx_len;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.part_o = static_cast<float*>(h->ws);
    p.part_ml = reinterpret_cast<float2*>(static_cast<char*>(h->ws) + pl.part_o_bytes);
    p.tickets = h->ctr;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const cudaError_t e = tt::launch_block_attn(maps, p, D, cs);
    if (e != cudaSuccess) return cuda_fail(e, "block attention launch");
    return TT_OK;
}

extern "C" {

int tt_block_attn(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                  const void* v_blk, const void* k_ctx, const void* v_ctx,
                  const int32_t* ctx_len, void* out, void* stream) {
    tt::TraceRange tr("tt_block_attn");
    return block_attn_call(h, d, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, out, stream, 0);
}

int tt_block_attn_causal(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                         const void* v_blk, const void* k_ctx, const void* v_ctx,
                         const int32_t* ctx_len, void* out, void* stream) {
    tt::TraceRange tr("tt_block_attn_causal");
    return block_attn_call(h, d, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, out, stream, 1);
}

int tt_block_attn_train(tt_handle h, const tt_train_desc* t, const void* q, const void* k_noisy,
                        const void* v_noisy, const void* k_clean, const void* v_clean, void* out,
                        void* stream) {
    tt::TraceRange tr("tt_block_attn_train");
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_block_attn_train: handle is NULL");
    tt_attn_desc d;
    const int st = train_desc(t, &d);
    if (st != TT_OK) return st;
    if (t->B == 0) return TT_OK;
    return block_attn_call(h, &d, q, k_noisy, v_noisy, k_clean, v_clean, nullptr, out, stream, 0,
                           t->N / t->S);
}

int tt_kv_append(tt_handle h, const tt_attn_desc* d, const void* k_blk, const void* v_blk,
                 void* k_ctx, void* v_ctx, int32_t* ctx_len, void* stream) {
    tt::TraceRange tr("tt_kv_append");
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_kv_append: handle is NULL");
    if (!d) return fail(TT_ERR_INVALID_ARG, "tt_kv_append: desc is NULL");
    if (d->B < 0 || d->B > 65535) return fail(TT_ERR_INVALID_ARG, "B=%d outside [0, 65535]", d->B);
    if (d->D != 64 && d->D != 128)
        return fail(TT_ERR_UNSUPPORTED, "head dim D=%d unsupported (64 or 128)", d->D);
    if (d->Hkv < 1 || d->Hkv > 65535) return fail(TT_ERR_INVALID_ARG, "Hkv=%d outside [1, 65535]", d->Hkv);
    if (d->ctx_cap < 1 || d->ctx_cap > (1 << 24))
        return fail(TT_ERR_INVALID_ARG, "ctx_cap=%d outside [1, 2^24]", d->ctx_cap);
    if (d->L < 1 || d->L > d->ctx_cap)
        return fail(TT_ERR_INVALID_ARG, "L=%d outside [1, ctx_cap=%d]", d->L, d->ctx_cap);
    if (d->B == 0) return TT_OK;
    if (!k_blk || !v_blk || !k_ctx || !v_ctx || !ctx_len)
        return fail(TT_ERR_INVALID_ARG, "tt_kv_append: a tensor pointer is NULL");
    if (!aligned16(k_blk) || !aligned16(v_blk) || !aligned16(k_ctx) || !aligned16(v_ctx) ||
        (reinterpret_cast<uintptr_t>(ctx_len) & 3u))
        return fail(TT_ERR_INVALID_ARG, "tt_kv_append: tensors must be 16-byte aligned");
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    tt::KvAppendParams p;
    p.B = d->B; p.L = d->L; p.Hkv = d->Hkv; p.D = d->D; p.ctx_cap = d->ctx_cap;
    p.k_blk = static_cast<const __nv_bfloat16*>(k_blk);
    p.v_blk = static_cast<const __nv_bfloat16*>(v_blk);
    p.k_ctx = static_cast<__nv_bfloat16*>(k_ctx);
    p.v_ctx = static_cast<__nv_bfloat16*>(v_ctx);
    p.ctx_len = ctx_len;
    p.status = h->status;
    const cudaError_t e = tt::launch_kv_append(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv append launch");
    return TT_OK;
}

int tt_commit_keys(tt_handle h, uint64_t* key_dst, int32_t* arg_dst, int rows, void* stream) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_commit_keys: handle is NULL");
    if (rows < 0) return fail(TT_ERR_INVALID_ARG, "tt_commit_keys: rows < 0");
    const size_t n = static_cast<size_t>(rows);
    if (commit_ws_bytes(n) > h->ws_bytes)
        return fail(TT_ERR_INVALID_ARG, "tt_commit_keys: more rows than the last commit held");
    if (n == 0) return TT_OK;
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (key_dst && (e = cudaMemcpyAsync(key_dst, h->ws, n * 8, cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "tt_commit_keys: copy keys");
    if (arg_dst &&
        (e = cudaMemcpyAsync(arg_dst, static_cast<char*>(h->ws) + align256(n * 8), n * 4,
                             cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "tt_commit_keys: copy predictions");
    return TT_OK;
}

}  // extern "C"

namespace {

// The largest key whose confidence 2^40 / key exceeds gamma, i.e. the largest
// integer key with gamma * key < 2^40, in exact arithmetic: gamma = M *
// 2^(e - 53) with an integer M (53 bits), so the condition is M * key <
// 2^(93 - e), decided on 128-bit integers. gamma <= 0: every key; gamma = +inf
// or a gamma that no key can meet: 0 (keys are >= 2^40).
unsigned long long key_threshold(double gamma) {
    if (!(gamma > 0.0)) return ~0ull;
    if (std::isinf(gamma)) return 0ull;
    int e = 0;
    const double f = std::frexp(gamma, &e);  // gamma = f * 2^e, f in [0.5, 1)
    const unsigned long long M = static_cast<unsigned long long>(std::ldexp(f, 53));  // exact
    const int sh = 93 - e;
    if (sh >= 127) return ~0ull;  // M * key < 2^110 <= 2^sh for every key
    if (sh <= 0) return 0ull;
    const unsigned __int128 lim = (static_cast<unsigned __int128>(1) << sh) - 1;
    const unsigned __int128 q = lim / M;
    return q > static_cast<unsigned __int128>(~0ull) ? ~0ull : static_cast<unsigned long long>(q);
}

int commit_impl(tt_handle h, const char* name, const float* logits, int B, int L, int V,
                const uint8_t* masked, int k, int steps_left, unsigned long long kthr,
                int32_t* tok, uint8_t* masked_out, void* stream) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "%s: handle is NULL", name);
    if (B < 0) return fail(TT_ERR_INVALID_ARG, "%s: B=%d < 0", name, B);
    if (L < 1 || L > tt::kCommitMaxL)
        return fail(TT_ERR_UNSUPPORTED, "%s: L=%d outside [1, %d]", name, L, tt::kCommitMaxL);
    if (V < 4 || V % 4 || V > tt::kCommitCluster * tt::kCommitSliceMax)
        return fail(TT_ERR_UNSUPPORTED, "%s: V=%d must be a multiple of 4 in [4, %d]", name, V,
                    tt::kCommitCluster * tt::kCommitSliceMax);
    if (static_cast<long>(B) * L > 0x7fffffffL / tt::kCommitCluster)
        return fail(TT_ERR_UNSUPPORTED, "%s: B*L too large", name);
    if (B == 0) return TT_OK;
    if (!logits || !masked || !tok || !masked_out)
        return fail(TT_ERR_INVALID_ARG, "%s: a tensor pointer is NULL", name);
    if (!aligned16(logits)) return fail(TT_ERR_INVALID_ARG, "%s: logits must be 16-byte aligned", name);
    if (!aligned16(tok)) return fail(TT_ERR_INVALID_ARG, "%s: tok must be 16-byte aligned", name);
    const size_t rows = static_cast<size_t>(B) * L;
    const uintptr_t mi = reinterpret_cast<uintptr_t>(masked), mo = reinterpret_cast<uintptr_t>(masked_out);
    if (mi != mo && mi < mo + rows && mo < mi + rows)
        return fail(TT_ERR_INVALID_ARG, "%s: masked and masked_out overlap without being the same buffer",
                    name);
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    int st = ensure_workspace(h, commit_ws_bytes(rows), 2 + static_cast<size_t>(B));
    if (st != TT_OK) return st;
    tt::CommitParams p;
    p.logits = logits;
    p.B = B; p.L = L; p.V = V; p.k = k;
    p.steps_left = steps_left;
    p.kthr = kthr;
    p.slice = (((V + tt::kCommitCluster - 1) / tt::kCommitCluster) + 3) & ~3;
    p.masked = masked;
    p.tok = tok;
    p.masked_out = masked_out;
    p.key = static_cast<unsigned long long*>(h->ws);
    p.arg = reinterpret_cast<int32_t*>(static_cast<char*>(h->ws) + align256(rows * 8));
    p.counters = h->ctr;
    p.alias = mi == mo;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    cudaError_t e = tt::launch_commit(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return TT_OK;
}

}  // namespace

extern "C" {

int tt_commit(tt_handle h, const float* logits, int B, int L, int V, const uint8_t* masked, int k,
              int32_t* tok, uint8_t* masked_out, void* stream) {
    tt::TraceRange tr("tt_commit");
    if (k < 1) return fail(TT_ERR_INVALID_ARG, "tt_commit: k=%d < 1", k);
    return commit_impl(h, "tt_commit", logits, B, L, V, masked, k, 0, 0ull, tok, masked_out, stream);
}

int tt_commit_threshold(tt_handle h, const float* logits, int B, int L, int V,
                        const uint8_t* masked, double gamma, int steps_left, int32_t* tok,
                        uint8_t* masked_out, void* stream) {
    tt::TraceRange tr("tt_commit_threshold");
    if (steps_left < 1)
        return fail(TT_ERR_INVALID_ARG, "tt_commit_threshold: steps_left=%d < 1", steps_left);
    if (std::isnan(gamma)) return fail(TT_ERR_INVALID_ARG, "tt_commit_threshold: gamma is NaN");
    return commit_impl(h, "tt_commit_threshold", logits, B, L, V, masked, 1, steps_left,
                       key_threshold(gamma), tok, masked_out, stream);
}

}  // extern "C"

// ---------------------------------------------------------------- LM head and the commit behind it
namespace {

// Grows the LM head's hand-off buffer (zeroed) to `rows` rows, with room for
// as many block tickets (a block has at least one row), so that the commit
// behind an LM head never has to grow it (growing clears the row maxima).
int ensure_lm(tt_context* h, size_t rows) {
    if (rows <= h->lm_rows) return TT_OK;
    const size_t r = rows, b = rows;
    cudaError_t e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (h->lm) cudaFree(h->lm);
    h->lm = nullptr;
    h->lm_rows = h->lm_blocks = 0;
    if ((e = cudaMalloc(&h->lm, r * 16 + b * 4)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(lm)");
    if ((e = cudaMemset(h->lm, 0, r * 16 + b * 4)) != cudaSuccess) return cuda_fail(e, "cudaMemset(lm)");
    h->lm_rows = r;
    h->lm_blocks = b;
    return TT_OK;
}

unsigned long long* lm_key(tt_context* h) { return static_cast<unsigned long long*>(h->lm); }
unsigned long long* lm_rowmax(tt_context* h) { return static_cast<unsigned long long*>(h->lm) + h->lm_rows; }
unsigned* lm_blk(tt_context* h) {
    return reinterpret_cast<unsigned*>(static_cast<unsigned long long*>(h->lm) + 2 * h->lm_rows);
}

int encode2d(tt_context* h, CUtensorMap* m, const void* base, int inner, int outer, int box_outer,
             const char* name) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t str[1] = {static_cast<cuuint64_t>(inner) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_outer)};
    return encode_cached(h, m, const_cast<void*>(base), 2, dims, str, box, name);
}

}  // namespace

extern "C" {

int tt_lm_head(tt_handle h, const void* hidden, const void* weight, int M, int K, int V, float* logits,
               void* stream) {
    tt::TraceRange tr("tt_lm_head");
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_lm_head: handle is NULL");
    if (M < 0 || K < 8 || K % 8 || V < 4 || V % 4)
        return fail(TT_ERR_INVALID_ARG, "tt_lm_head: needs M >= 0, K >= 8 with K %% 8 == 0, V >= 4 with V %% 4 == 0");
    if (K > (1 << 20) || V > (1 << 24) || M > (1 << 24))
        return fail(TT_ERR_UNSUPPORTED, "tt_lm_head: K, V or M too large");
    if (M == 0) return TT_OK;
    if (!hidden || !weight || !logits) return fail(TT_ERR_INVALID_ARG, "tt_lm_head: a tensor pointer is NULL");
    if (!aligned16(hidden) || !aligned16(weight) || !aligned16(logits))
        return fail(TT_ERR_INVALID_ARG, "tt_lm_head: tensors must be 16-byte aligned");
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    int st = ensure_lm(h, static_cast<size_t>(M));
    if (st != TT_OK) return st;
    CUtensorMap ma, mb;
    if ((st = encode2d(h, &ma, hidden, K, M, 128, "hidden")) != TT_OK) return st;
    if ((st = encode2d(h, &mb, weight, K, V, 256, "weight")) != TT_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    // each row's maximum is an atomic max over the vocabulary tiles: from zero
    if ((e = cudaMemsetAsync(lm_rowmax(h), 0, static_cast<size_t>(M) * 8, s)) != cudaSuccess)
        return cuda_fail(e, "tt_lm_head: clear row maxima");
    tt::LmHeadParams p;
    p.M = M; p.K = K; p.V = V;
    p.logits = logits;
    p.rowmax = lm_rowmax(h);
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    if ((e = tt::launch_lm_head(ma, mb, p, h->num_sms, s)) != cudaSuccess)
        return cuda_fail(e, "tt_lm_head launch");
    h->lm_M = M;
    h->lm_V = V;
    return TT_OK;
}

static int commit_rowmax_impl(tt_handle h, const char* name, const float* logits, int B, int L, int V,
                              const uint8_t* masked, int k, int steps_left, unsigned long long kthr,
                              int32_t* tok, uint8_t* masked_out, void* stream) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "%s: handle is NULL", name);
    if (B < 0 || L < 1 || L > tt::kCommitMaxL)
        return fail(TT_ERR_INVALID_ARG, "%s: needs B >= 0 and 1 <= L <= %d", name, tt::kCommitMaxL);
    if (B == 0) return TT_OK;
    if (static_cast<long long>(B) * L != h->lm_M || V != h->lm_V)
        return fail(TT_ERR_INVALID_ARG, "%s: B*L and V must be the M and V of the last tt_lm_head call", name);
    if (!logits || !masked || !tok || !masked_out)
        return fail(TT_ERR_INVALID_ARG, "%s: a tensor pointer is NULL", name);
    if (!aligned16(logits)) return fail(TT_ERR_INVALID_ARG, "%s: logits must be 16-byte aligned", name);
    const size_t rows = static_cast<size_t>(B) * L;
    const uintptr_t mi = reinterpret_cast<uintptr_t>(masked), mo = reinterpret_cast<uintptr_t>(masked_out);
    if (mi != mo && mi < mo + rows && mo < mi + rows)
        return fail(TT_ERR_INVALID_ARG, "%s: masked and masked_out overlap without being the same buffer", name);
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    int st = ensure_lm(h, rows);  // no growth: rows == the LM head's M
    if (st != TT_OK) return st;
    if ((st = ensure_workspace(h, commit_ws_bytes(rows), 0)) != TT_OK) return st;
    tt::RowmaxCommitParams p;
    p.logits = logits;
    p.B = B; p.L = L; p.V = V; p.k = k;
    p.steps_left = steps_left;
    p.kthr = kthr;
    p.masked = masked;
    p.tok = tok;
    p.masked_out = masked_out;
    p.key = lm_key(h);
    p.rowmax = lm_rowmax(h);
    p.blk = lm_blk(h);
    p.key_out = static_cast<unsigned long long*>(h->ws);
    p.arg = reinterpret_cast<int32_t*>(static_cast<char*>(h->ws) + align256(rows * 8));
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    const cudaError_t e = tt::launch_commit_rowmax(p, h->num_sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return TT_OK;
}

int tt_commit_rowmax(tt_handle h, const float* logits, int B, int L, int V, const uint8_t* masked, int k,
                     int32_t* tok, uint8_t* masked_out, void* stream) {
    tt::TraceRange tr("tt_commit_rowmax");
    if (k < 1) return fail(TT_ERR_INVALID_ARG, "tt_commit_rowmax: k=%d < 1", k);
    return commit_rowmax_impl(h, "tt_commit_rowmax", logits, B, L, V, masked, k, 0, 0ull, tok, masked_out,
                              stream);
}

}  // extern "C"
