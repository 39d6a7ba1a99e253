// C-ABI layer: argument checks, launch planning (KV splits), TMA tensor-map
// encoding and kernel launches. See include/tt.h for the contract.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "tt.h"
#include "tt_internal.h"

struct tt_context {
    int device;
    int num_sms;
    unsigned* status;  // device word, TT_DEV_* bits
    unsigned long long timeout_ns;
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
    int G, n_mtiles, n_pairs, nblk, nt_max, splits, chunk;
    size_t ws_o_bytes, ws_bytes;
};

// Checks a descriptor; fills the launch plan. Split choice: minimise
// waves * (tiles per split + 2) over the split count, where one wave is one
// CTA per SM (the kernel's shared memory allows one) and the +2 stands for the
// per-CTA prologue and epilogue; a split sequence also pays for the merge.
int plan_attn(const tt_attn_desc* d, int num_sms, AttnPlan* pl) {
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
    if (d->num_splits < 0) return fail(TT_ERR_INVALID_ARG, "num_splits must be >= 0");
    pl->G = G;
    pl->n_mtiles = static_cast<int>((static_cast<long>(G) * d->L + tt::kTile - 1) / tt::kTile);
    pl->n_pairs = (pl->n_mtiles + 1) / 2;
    pl->nblk = (d->L + tt::kTile - 1) / tt::kTile;
    pl->nt_max = (d->ctx_cap + tt::kTile - 1) / tt::kTile + pl->nblk;
    const long units = static_cast<long>(d->B) * d->Hkv * pl->n_pairs;
    int best = 1;
    if (d->num_splits > 0) {
        best = d->num_splits < pl->nt_max ? d->num_splits : pl->nt_max;
    } else if (units > 0) {
        double best_cost = 1e300;
        const int smax = pl->nt_max < 64 ? pl->nt_max : 64;
        for (int s = 1; s <= smax; ++s) {
            const int chunk = (pl->nt_max + s - 1) / s;
            const int s2 = (pl->nt_max + chunk - 1) / chunk;
            if (s2 != s) continue;
            const long waves = (units * s2 + num_sms - 1) / num_sms;
            const double cost = static_cast<double>(waves) * (chunk + 2) + (s2 > 1 ? 2 : 0);
            if (cost < best_cost) { best_cost = cost; best = s2; }
        }
    }
    pl->chunk = (pl->nt_max + best - 1) / best;
    pl->splits = (pl->nt_max + pl->chunk - 1) / pl->chunk;
    if (pl->splits > 1) {
        const size_t rows = static_cast<size_t>(pl->splits) * d->B * d->Hkv *
                            static_cast<size_t>(pl->n_mtiles) * tt::kTile;
        pl->ws_o_bytes = align256(rows * d->D * sizeof(float));
        pl->ws_bytes = pl->ws_o_bytes + align256(rows * 2 * sizeof(float));
    } else {
        pl->ws_o_bytes = pl->ws_bytes = 0;
    }
    const long grid_x = static_cast<long>(pl->n_pairs) * pl->splits;
    if (grid_x > 0x7fffffffL) return fail(TT_ERR_UNSUPPORTED, "grid too large");
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

}  // namespace

void tt::record_host_error(const char* where, const char* msg) { fail(0, "%s: %s", where, msg); }

extern "C" {

const char* tt_status_string(int s) {
    switch (s) {
        case TT_OK: return "TT_OK";
        case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG";
        case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED";
        case TT_ERR_CUDA: return "TT_ERR_CUDA";
        case TT_ERR_DEVICE: return "TT_ERR_DEVICE";
        case TT_ERR_WORKSPACE: return "TT_ERR_WORKSPACE";
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
    if ((e = tt::configure_commit_kernels()) != cudaSuccess) return cuda_fail(e, "commit kernel attributes");
    tt_context* h = new tt_context();
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    h->timeout_ns = 1000000000ull;
    if ((e = cudaMalloc(&h->status, sizeof(unsigned))) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaMalloc(status)");
    }
    if ((e = cudaMemset(h->status, 0, sizeof(unsigned))) != cudaSuccess) {
        cudaFree(h->status);
        delete h;
        return cuda_fail(e, "cudaMemset(status)");
    }
    *out = h;
    return TT_OK;
}

int tt_destroy(tt_handle h) {
    if (!h) return TT_OK;
    DeviceGuard g(h->device);
    cudaFree(h->status);
    delete h;
    return TT_OK;
}

int tt_set_wait_timeout(tt_handle h, unsigned long long ns) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "handle is NULL");
    if (ns == 0) return fail(TT_ERR_INVALID_ARG, "timeout must be > 0");
    h->timeout_ns = ns;
    return TT_OK;
}

int tt_get_error(tt_handle h, unsigned* device_status) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "handle is NULL");
    DeviceGuard g(h->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned v = 0;
    if ((e = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "read status");
    if ((e = cudaMemset(h->status, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "clear status");
    if (device_status) *device_status = v;
    return v ? TT_ERR_DEVICE : TT_OK;
}

size_t tt_block_attn_workspace_bytes(tt_handle h, const tt_attn_desc* d) {
    if (!h) return 0;
    AttnPlan pl;
    if (plan_attn(d, h->num_sms, &pl) != TT_OK) return 0;
    return pl.ws_bytes;
}

// Body of tt_block_attn (causal = 0), tt_block_attn_causal (causal = 1) and
// tt_block_attn_train (ctx_group = blocks per clean sequence: d->B counts the
// noisy blocks, the caches belong to d->B / ctx_group clean sequences and
// ctx_len is implied).
static int block_attn_call(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                           const void* v_blk, const void* k_ctx, const void* v_ctx,
                           const int32_t* ctx_len, void* out, void* workspace,
                           size_t workspace_bytes, void* stream, int causal, int ctx_group = 0) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_block_attn: handle is NULL");
    AttnPlan pl;
    int st = plan_attn(d, h->num_sms, &pl);
    if (st != TT_OK) return st;
    if (d->B == 0) return TT_OK;
    if (!q || !k_blk || !v_blk || (!ctx_len && !ctx_group) || !out)
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: a tensor pointer is NULL");
    if (d->ctx_cap > 0 && (!k_ctx || !v_ctx))
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: k_ctx/v_ctx NULL with ctx_cap > 0");
    if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out) ||
        (d->ctx_cap > 0 && (!aligned16(k_ctx) || !aligned16(v_ctx))))
        return fail(TT_ERR_INVALID_ARG, "tt_block_attn: tensors must be 16-byte aligned");
    if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes ||
                            (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(TT_ERR_WORKSPACE, "tt_block_attn: needs %zu workspace bytes (256-byte aligned)",
                    pl.ws_bytes);
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);

    const int B = d->B, L = d->L, Hq = d->Hq, Hkv = d->Hkv, D = d->D, G = pl.G;
    const cuuint64_t e2 = 2;  // bytes per bf16
    tt::AttnMaps maps;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)Hkv, (cuuint64_t)L,
                                    (cuuint64_t)B};
        const cuuint64_t str[4] = {D * e2, (cuuint64_t)G * D * e2, (cuuint64_t)Hq * D * e2,
                                   (cuuint64_t)L * Hq * D * e2};
        const cuuint32_t box[5] = {64, (cuuint32_t)G, 1, (cuuint32_t)(tt::kTile / G), 1};
        if ((st = encode(&maps.q, const_cast<void*>(q), 5, dims, str, box, "q")) != TT_OK) return st;
    }
    {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)L, (cuuint64_t)B};
        const cuuint64_t str[3] = {D * e2, (cuuint64_t)Hkv * D * e2, (cuuint64_t)L * Hkv * D * e2};
        const cuuint32_t box[4] = {64, 1, (cuuint32_t)tt::kTile, 1};
        if ((st = encode(&maps.k_blk, const_cast<void*>(k_blk), 4, dims, str, box, "k_blk")) != TT_OK)
            return st;
        if ((st = encode(&maps.v_blk, const_cast<void*>(v_blk), 4, dims, str, box, "v_blk")) != TT_OK)
            return st;
    }
    {
        // With no cache (ctx_cap == 0) no context tile is ever loaded; the maps
        // only need to be well formed, so they point at the block keys.
        const bool none = d->ctx_cap == 0;
        const cuuint64_t dims[3] = {(cuuint64_t)D, none ? (cuuint64_t)tt::kTile : (cuuint64_t)d->ctx_cap,
                                    none ? 1 : (cuuint64_t)(ctx_group ? B / ctx_group : B) * Hkv};
        const cuuint64_t str[2] = {D * e2, (none ? (cuuint64_t)tt::kTile : (cuuint64_t)d->ctx_cap) * D * e2};
        const cuuint32_t box[3] = {64, (cuuint32_t)tt::kTile, 1};
        void* kc = none ? const_cast<void*>(k_blk) : const_cast<void*>(k_ctx);
        void* vc = none ? const_cast<void*>(v_blk) : const_cast<void*>(v_ctx);
        if ((st = encode(&maps.k_ctx, kc, 3, dims, str, box, "k_ctx")) != TT_OK) return st;
        if ((st = encode(&maps.v_ctx, vc, 3, dims, str, box, "v_ctx")) != TT_OK) return st;
    }
    tt::AttnParams p;
    p.B = B; p.L = L; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.ctx_cap = d->ctx_cap;
    p.n_mtiles = pl.n_mtiles; p.n_pairs = pl.n_pairs; p.chunk = pl.chunk; p.nblk = pl.nblk;
    p.causal = causal;
    p.ctx_group = ctx_group;
    const float scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(D));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.ctx_len = ctx_len;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.ws_o = pl.splits > 1 ? static_cast<float*>(workspace) : nullptr;
    p.ws_ml = pl.splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.ws_o_bytes)
                            : nullptr;
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = tt::launch_block_attn(maps, p, D, pl.splits, s);
    if (e != cudaSuccess) return cuda_fail(e, "block attention launch");
    if (pl.splits > 1) {
        e = tt::launch_attn_merge(p, D, s);
        if (e != cudaSuccess) return cuda_fail(e, "split merge launch");
    }
    return TT_OK;
}

int tt_block_attn(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                  const void* v_blk, const void* k_ctx, const void* v_ctx,
                  const int32_t* ctx_len, void* out, void* workspace, size_t workspace_bytes,
                  void* stream) {
    return block_attn_call(h, d, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, out, workspace,
                           workspace_bytes, stream, 0);
}

int tt_block_attn_causal(tt_handle h, const tt_attn_desc* d, const void* q, const void* k_blk,
                         const void* v_blk, const void* k_ctx, const void* v_ctx,
                         const int32_t* ctx_len, void* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return block_attn_call(h, d, q, k_blk, v_blk, k_ctx, v_ctx, ctx_len, out, workspace,
                           workspace_bytes, stream, 1);
}

// Checks a training-layout descriptor and gives the equivalent per-block one.
static int train_desc(const tt_train_desc* t, tt_attn_desc* d) {
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
    d->num_splits = t->num_splits;
    return TT_OK;
}

size_t tt_block_attn_train_workspace_bytes(tt_handle h, const tt_train_desc* t) {
    tt_attn_desc d;
    if (!h || train_desc(t, &d) != TT_OK) return 0;
    AttnPlan pl;
    if (plan_attn(&d, h->num_sms, &pl) != TT_OK) return 0;
    return pl.ws_bytes;
}

int tt_block_attn_train(tt_handle h, const tt_train_desc* t, const void* q, const void* k_noisy,
                        const void* v_noisy, const void* k_clean, const void* v_clean, void* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
    if (!h) return fail(TT_ERR_INVALID_ARG, "tt_block_attn_train: handle is NULL");
    tt_attn_desc d;
    const int st = train_desc(t, &d);
    if (st != TT_OK) return st;
    if (t->B == 0) return TT_OK;
    return block_attn_call(h, &d, q, k_noisy, v_noisy, k_clean, v_clean, nullptr, out, workspace,
                           workspace_bytes, stream, 0, t->N / t->S);
}

int tt_kv_append(tt_handle h, const tt_attn_desc* d, const void* k_blk, const void* v_blk,
                 void* k_ctx, void* v_ctx, int32_t* ctx_len, void* stream) {
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

size_t tt_commit_workspace_bytes(int B, int L) {
    if (B < 0 || L < 0) return 0;
    const size_t rows = static_cast<size_t>(B) * L;
    return align256(rows * 8) + align256(rows * 4) + static_cast<size_t>(B) * 4;
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
                int32_t* tok, uint8_t* masked_out, void* workspace, size_t workspace_bytes,
                void* stream) {
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
    const size_t need = tt_commit_workspace_bytes(B, L);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(TT_ERR_WORKSPACE, "%s: needs %zu workspace bytes (256-byte aligned)", name, need);
    DeviceGuard g(h->device);
    if (!g.ok()) return fail(TT_ERR_CUDA, "cannot select device %d", h->device);
    tt::CommitParams p;
    p.logits = logits;
    p.B = B; p.L = L; p.V = V; p.k = k;
    p.steps_left = steps_left;
    p.kthr = kthr;
    p.slice = (((V + tt::kCommitCluster - 1) / tt::kCommitCluster) + 3) & ~3;
    p.masked = masked;
    p.tok = tok;
    p.masked_out = masked_out;
    p.key = static_cast<unsigned long long*>(workspace);
    const size_t rows = static_cast<size_t>(B) * L;
    p.arg = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + align256(rows * 8));
    p.counters = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + align256(rows * 8) +
                                             align256(rows * 4));
    p.status = h->status;
    p.timeout_ns = h->timeout_ns;
    cudaError_t e = tt::launch_commit(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return TT_OK;
}

}  // namespace

extern "C" {

int tt_commit(tt_handle h, const float* logits, int B, int L, int V, const uint8_t* masked, int k,
              int32_t* tok, uint8_t* masked_out, void* workspace, size_t workspace_bytes,
              void* stream) {
    if (k < 1) return fail(TT_ERR_INVALID_ARG, "tt_commit: k=%d < 1", k);
    return commit_impl(h, "tt_commit", logits, B, L, V, masked, k, 0, 0ull, tok, masked_out,
                       workspace, workspace_bytes, stream);
}

int tt_commit_threshold(tt_handle h, const float* logits, int B, int L, int V,
                        const uint8_t* masked, double gamma, int steps_left, int32_t* tok,
                        uint8_t* masked_out, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (steps_left < 1)
        return fail(TT_ERR_INVALID_ARG, "tt_commit_threshold: steps_left=%d < 1", steps_left);
    if (std::isnan(gamma)) return fail(TT_ERR_INVALID_ARG, "tt_commit_threshold: gamma is NaN");
    return commit_impl(h, "tt_commit_threshold", logits, B, L, V, masked, 1, steps_left,
                       key_threshold(gamma), tok, masked_out, workspace, workspace_bytes, stream);
}

}  // extern "C"
