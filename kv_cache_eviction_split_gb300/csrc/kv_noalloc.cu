// kv_noalloc.cu -- kv_score for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// where the CUDA allocator must not be called after start-up (a serving
// process that reserves all device memory up front, a plugin inside a host
// application that owns the allocator, a latency-critical path that forbids
// cudaMalloc and its implicit synchronisation).  kv_score_noalloc gives them
// the scoring step with its scratch in one fixed array of this library's own
// device memory instead of a caller workspace.
//
// The array is kNoAllocScratchBytes (64 MiB).  Every GPU that loads this
// library holds it until the process exits.  Problems whose kv_score
// workspace would exceed it are rejected with KV_ERR_WORKSPACE.  All calls
// share the one array and it keeps the last call's contents: calls whose work
// overlaps on the GPU (different streams, or different host threads on the same
// device) race on it.
//
// The array's device address belongs to a CUDA context: the module that holds
// it is loaded again into a new context after cudaDeviceReset, or into another
// context made current on the same device.  The address is therefore cached
// per context, keyed on the context's unique ID (cuCtxGetId), and looked up
// again with cudaGetSymbolAddress whenever the current context is one not seen
// before.
#include <cudaTypedefs.h>

#include <mutex>

#include "kv_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// File-scope scratch; host code must not use its name as a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    unsigned long long ctx_id;   // unique ID of the context the address belongs to
    void *addr;
};
Cached g_cache[kMaxDevices] = {};

// Driver entry points (through the runtime, so the library links no libcuda).
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns &ctx_fns() {
    static const CtxFns fns = [] {
        CtxFns f;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        return f;
    }();
    return fns;
}

// Unique ID of the current context; false if there is none (or it cannot be read).
bool current_ctx_id(unsigned long long *id) {
    const CtxFns &f = ctx_fns();
    if (!f.get_current || !f.get_id) return false;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return f.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context.
kv_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned long long id = 0;
    if (current_ctx_id(&id) && g_cache[dev].addr && g_cache[dev].ctx_id == id) {
        *out = g_cache[dev].addr;
        return KV_OK;
    }
    // first call in this context (the lookup also makes the device's primary
    // context current if none was)
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KV_ERR_CUDA;
    if (!current_ctx_id(&id)) return KV_ERR_CUDA;
    g_cache[dev] = {id, p};
    *out = p;
    return KV_OK;
}

}  // namespace

extern "C" kv_status kv_score_noalloc(const kv_problem *p, const void *q_win, const void *k,
                                      const void *v, float *scores, void *stream) {
    size_t need = 0;
    kv_status st = kv_score_workspace_size(p, &need);
    if (st != KV_OK) return st;
    if (need > kNoAllocScratchBytes) return KV_ERR_WORKSPACE;
    if (p->num_requests == 0) return KV_OK;
    void *ws = nullptr;
    st = scratch_address(&ws);
    if (st != KV_OK) return st;
    // the header (status words) must start at zero
    if (cudaMemsetAsync(ws, 0, kvevict::kHeaderBytes, (cudaStream_t)stream) != cudaSuccess)
        return KV_ERR_CUDA;
    return kv_score(p, q_win, k, v, scores, ws, kNoAllocScratchBytes, stream);
}
