// kv_score.cu -- the stand-alone split-K merge kernel (merge_row in
// kv_merge.cuh) and the launcher of pass 1 + merge.
#include "kv_merge.cuh"

namespace kvevict {
namespace {

template <int D, bool kO>
__global__ void __launch_bounds__(128)
attn_merge_kernel(DevProblem P, ScoreWs ws) {
    const int row = blockIdx.y * 4 + (threadIdx.x >> 5);
    if (row < ws.a_rows) merge_row<D, kO>(P, ws, blockIdx.x, row, threadIdx.x & 31);
}

template <int D>
cudaError_t merge_d(const DevProblem &P, const ScoreWs &ws, cudaStream_t st) {
    dim3 g((unsigned)P.units, (ws.a_rows + 3) / 4);
    if (P.rule == KV_SCORE_ATTN_SUM)
        attn_merge_kernel<D, false><<<g, 128, 0, st>>>(P, ws);
    else
        attn_merge_kernel<D, true><<<g, 128, 0, st>>>(P, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t s) {
    cudaError_t e = launch_attention_partials(P, q, k, v, ws, s);
    if (e != cudaSuccess) return e;
    return P.d == 64 ? merge_d<64>(P, ws, s) : merge_d<128>(P, ws, s);
}

}  // namespace kvevict
