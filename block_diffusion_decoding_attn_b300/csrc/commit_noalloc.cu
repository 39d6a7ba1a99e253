// tt_commit_noalloc: the unmask/commit step for callers that cannot allocate
// device memory. A serving engine that reserves all of HBM for its own pool
// when it starts, or a plug-in host that forbids allocation while a request
// runs, can call neither cudaMalloc nor any allocating library routine, and
// may not be able to hand out a zero-filled workspace either. This entry
// point keeps the commit step's scratch (per-row keys and predictions,
// per-block tickets) in a fixed array compiled into the library instead.
//
// The array holds kScratchBytes (about 1 MiB) on every GPU that loads
// the library, until the process exits; it bounds B*L to 65536 rows. Every
// call uses the same array, so calls whose work overlaps on the GPU (other
// streams, other host threads) race on it and must be ordered by the caller.
#include <mutex>

#include "host_trace.h"
#include "tt.h"
#include "tt_internal.h"

namespace {

constexpr int kMaxRows = 65536;    // B * L
constexpr int kMaxBlocks = 65536;  // B
constexpr size_t kKeyOff = 0;                                                    // uint64 key[kMaxRows]
constexpr size_t kArgOff = kKeyOff + static_cast<size_t>(kMaxRows) * 8;          // int32 arg[kMaxRows]
// uint32 counters[2 + kMaxBlocks]: two per-call counters, then the block tickets
constexpr size_t kTicketOff = kArgOff + static_cast<size_t>(kMaxRows) * 4;
constexpr size_t kStatusOff = kTicketOff + static_cast<size_t>(2 + kMaxBlocks) * 4;  // uint32 status
constexpr size_t kScratchBytes = kStatusOff + 256;

// In host code this name is only a stand-in for the device array, not its
// address: the device address comes from cudaGetSymbolAddress (below), looked
// up once per device with that device current.
static __device__ __align__(256) unsigned char g_commit_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char* g_scratch_dev[kMaxDevices] = {};

int fail(int status, const char* msg) {
    tt::record_host_error("tt_commit_noalloc", msg);  // read back with tt_last_error()
    return status;
}

}  // namespace

extern "C" int tt_commit_noalloc(const float* logits, int B, int L, int V, const uint8_t* masked,
                                 int k, int32_t* tok, uint8_t* masked_out, void* stream) {
    tt::TraceRange tr("tt_commit_noalloc");
    if (B < 0 || L < 1 || k < 1) return fail(TT_ERR_INVALID_ARG, "needs B >= 0, L >= 1, k >= 1");
    if (static_cast<long>(B) * L > kMaxRows || B > kMaxBlocks)
        return fail(TT_ERR_UNSUPPORTED,
                    "B*L exceeds 65536 rows, the size of the built-in scratch; use tt_commit");
    if (L > tt::kCommitMaxL) return fail(TT_ERR_UNSUPPORTED, "L exceeds 16384");
    if (V < 4 || V % 4 || V > tt::kCommitCluster * tt::kCommitSliceMax)
        return fail(TT_ERR_UNSUPPORTED, "V must be a multiple of 4 in [4, 131072]");
    if (B == 0) return TT_OK;
    if (!logits || !masked || !tok || !masked_out)
        return fail(TT_ERR_INVALID_ARG, "a tensor pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(logits) & 15u) || (reinterpret_cast<uintptr_t>(tok) & 15u))
        return fail(TT_ERR_INVALID_ARG, "logits and tok must be 16-byte aligned");
    const uintptr_t mi = reinterpret_cast<uintptr_t>(masked), mo = reinterpret_cast<uintptr_t>(masked_out);
    const size_t rows = static_cast<size_t>(B) * L;
    if (mi != mo && mi < mo + rows && mo < mi + rows)
        return fail(TT_ERR_INVALID_ARG, "masked and masked_out overlap without being the same buffer");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(TT_ERR_CUDA, "no usable current CUDA device");
    unsigned char* base;
    {
        // Set-up on the first call on this device (the current one): the
        // array's device address and the commit kernel's launch attributes.
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_scratch_dev[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_commit_scratch) != cudaSuccess || !ptr)
                return fail(TT_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed");
            if (tt::configure_commit_kernels() != cudaSuccess)
                return fail(TT_ERR_CUDA, "setting the commit kernel's attributes failed");
            g_scratch_dev[dev] = static_cast<unsigned char*>(ptr);
        }
        base = g_scratch_dev[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents. The counters and block
    // tickets must start at zero (a call that gave up on a wait may have left
    // them otherwise), so they are cleared; the keys and predictions are
    // written before they are read.
    if (cudaMemsetAsync(base + kTicketOff, 0, static_cast<size_t>(2 + B) * 4, s) != cudaSuccess)
        return fail(TT_ERR_CUDA, "clearing the block tickets failed");
    tt::CommitParams p;
    p.logits = logits;
    p.B = B;
    p.L = L;
    p.V = V;
    p.k = k;
    p.steps_left = 0;  // fixed budget of k
    p.kthr = 0;
    p.slice = (((V + tt::kCommitCluster - 1) / tt::kCommitCluster) + 3) & ~3;  // per-CTA share
    p.masked = masked;
    p.tok = tok;
    p.masked_out = masked_out;
    p.key = reinterpret_cast<unsigned long long*>(base + kKeyOff);
    p.arg = reinterpret_cast<int32_t*>(base + kArgOff);
    p.counters = reinterpret_cast<unsigned*>(base + kTicketOff);
    p.alias = mi == mo;
    p.status = reinterpret_cast<unsigned*>(base + kStatusOff);
    p.timeout_ns = 1000000000ull;
    if (tt::launch_commit(p, s) != cudaSuccess) return fail(TT_ERR_CUDA, "commit launch failed");
    return TT_OK;
}

extern "C" int tt_commit_noalloc_status(int* device_status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(TT_ERR_CUDA, "no usable current CUDA device");
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_scratch_dev[dev])
            return fail(TT_ERR_INVALID_ARG, "no tt_commit_noalloc call was made on this device");
    }
    unsigned v = 0;
    const unsigned zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(TT_ERR_CUDA, "cudaDeviceSynchronize failed");
    // Synchronous copies of the status word inside the built-in array.
    if (cudaMemcpyFromSymbol(&v, g_commit_scratch, sizeof v, kStatusOff) != cudaSuccess)
        return fail(TT_ERR_CUDA, "reading the status word failed");
    if (cudaMemcpyToSymbol(g_commit_scratch, &zero, sizeof zero, kStatusOff) != cudaSuccess)
        return fail(TT_ERR_CUDA, "clearing the status word failed");
    if (device_status) *device_status = static_cast<int>(v);
    return (v & tt::kDevWaitTimeout) ? TT_ERR_TIMEOUT : TT_OK;
}
