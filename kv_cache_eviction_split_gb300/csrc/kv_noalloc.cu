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
// overlaps on the GPU (different streams, or different host threads on the
// same device) race on it.
#include <mutex>

#include "kv_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// File-scope scratch; host code must not use its name as a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
kv_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KV_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
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
    // the status word at the head of the workspace must start at zero
    if (cudaMemsetAsync(ws, 0, kvevict::kHeaderBytes, (cudaStream_t)stream) != cudaSuccess)
        return KV_ERR_CUDA;
    return kv_score(p, q_win, k, v, scores, ws, kNoAllocScratchBytes, stream);
}
