// kv_common.cu -- helpers shared by the two scoring passes: the per-unit work
// plan (prefix sums of key blocks, for ragged request lengths) and TMA maps.
#include <cudaTypedefs.h>

#include "kv_internal.cuh"

namespace kvevict {
namespace {

__global__ void __launch_bounds__(1024) plan_kernel(DevProblem P, int keys_per_block,
                                                    int32_t *plan) {
    __shared__ int32_t warp_sums[32];
    const long long U = P.units;
    const long long per = (U + blockDim.x - 1) / blockDim.x;
    const long long u0 = threadIdx.x * per, u1 = min(U, u0 + per);
    auto blocks_of = [&](long long u) {
        const int r = (int)(u / ((long long)P.L * P.H));
        const int n = (int)(P.cu[r + 1] - P.cu[r]);
        return (n + keys_per_block - 1) / keys_per_block;
    };
    int32_t mine = 0;
    for (long long u = u0; u < u1; ++u) mine += blocks_of(u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = mine;
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t t = warp_sums[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        warp_sums[lane] = t;
    }
    __syncthreads();
    int32_t run = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - mine;
    for (long long u = u0; u < u1; ++u) {
        plan[u] = run;
        run += blocks_of(u);
    }
    if (threadIdx.x == blockDim.x - 1) plan[U] = run;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

}  // namespace

void launch_plan(const DevProblem &P, int keys_per_block, int32_t *plan, cudaStream_t s) {
    plan_kernel<<<1, 1024, 0, s>>>(P, keys_per_block, plan);
}

long long total_blocks(const DevProblem &P, int keys_per_block) {
    long long blocks = 0;
    for (long long u = 0; u < P.units; ++u) {
        const int r = (int)(u / ((long long)P.L * P.H));
        const long long n = P.host_cu[r + 1] - P.host_cu[r];
        blocks += (n + keys_per_block - 1) / keys_per_block;
    }
    return blocks;
}

bool make_tile_map(CUtensorMap *m, const void *base, long long rows, int D) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvevict
