// kv_select.cu -- the stand-alone budgeted top-k: one 1024-thread CTA per unit
// runs select_unit (kv_select.cuh).
#include "kv_select.cuh"

namespace kvevict {
namespace {

constexpr int kSelThreads = 1024;

__global__ void __launch_bounds__(kSelThreads)
select_kernel(DevProblem P, const float *__restrict__ scores, const int32_t *__restrict__ budgets,
              const int64_t *__restrict__ offsets, int32_t *__restrict__ sel, int *status) {
    __shared__ unsigned smem[sel_smem_bytes<kSelThreads>() / 4];
    select_unit<kSelThreads, false, 16>(P, scores, budgets, offsets, sel, status, blockIdx.x,
                                        sel_smem<kSelThreads>(smem));
}

}  // namespace

cudaError_t launch_select(const DevProblem &P, const float *scores, const int32_t *budgets,
                          const int64_t *offsets, int32_t *sel, int *status, cudaStream_t s) {
    select_kernel<<<(unsigned)P.units, kSelThreads, 0, s>>>(P, scores, budgets, offsets, sel,
                                                            status);
    return cudaGetLastError();
}

}  // namespace kvevict
