// kv_attention.cu -- the stand-alone pass-1 kernels (bodies in kv_pass1.cuh)
// and their launcher: attn_tc_kernel for the DropKV rules, attn_stats_kernel
// (row statistics from K alone) for the attention sum.
#include <algorithm>

#include "kv_pass1.cuh"

namespace kvevict {
namespace {
using namespace sm100;
using namespace pass1;

template <int D, bool kOneQ>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const AttnArgs A, const __grid_constant__ ItemOrder ord) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t tmem =
        tmem_acquire_all(reinterpret_cast<uint32_t *>(smem + Layout<D, kOneQ>::kMisc));
    attn_tc_body<D, kOneQ>(P, &tm_q, &tm_k, &tm_v, A, ord, smem, tmem, blockIdx.x, gridDim.x);
    tmem_release_all(tmem);
}

template <int D>
__global__ void __launch_bounds__(kStatThreads, 1)
attn_stats_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const AttnArgs A,
                  const __grid_constant__ ItemOrder ord) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t tmem =
        tmem_acquire_all(reinterpret_cast<uint32_t *>(smem + StatLayout<D>::kMisc));
    attn_stats_body<D>(P, &tm_q, &tm_k, A, ord, smem, tmem, blockIdx.x, gridDim.x);
    tmem_release_all(tmem);
}

template <int D>
cudaError_t attention_d(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                        const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const long long q_rows = (long long)P.R * P.L * P.Hq * P.w;
    const long long kv_rows = (long long)P.L * P.H * P.N_tot;
    if (!make_tile_map(&mq, q, q_rows, D) || !make_tile_map(&mk, k, kv_rows, D) ||
        !make_tile_map(&mv, v, kv_rows, D))
        return cudaErrorInvalidValue;
    ItemOrder ord;
    build_item_order(P, P.split_keys, &ord);
    if (ord.nrun == 0)   // only with more runs of lengths than the order tables hold
        launch_plan(P, P.split_keys, ws.plan, st);
    AttnArgs A;
    A.plan = ws.plan;
    A.part_ml = ws.part_ml;
    A.part_o = ws.part_o;
    A.v2 = ws.v2;
    A.chunks = ws.chunks;
    A.parts = ws.parts;
    A.pairs = ws.parts == 1 ? (ws.chunks + 1) / 2 : 1;
    A.total_items = total_blocks(P, P.split_keys) * A.pairs;
    A.status = ws.status;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long grid = std::min<long long>(sms, A.total_items);
    if (P.rule == KV_SCORE_ATTN_SUM) {
        const int smem = StatLayout<D>::kTotal;
        cudaFuncSetAttribute(attn_stats_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
        if (grid > 0)
            attn_stats_kernel<D><<<(unsigned)grid, kStatThreads, smem, st>>>(P, mq, mk, A, ord);
        return cudaGetLastError();
    }
    // one row chunk (lanes on alternate tiles): one Q slot and a third V stage
    if (A.parts == 2) {
        const int smem = Layout<D, true>::kTotal;
        cudaFuncSetAttribute(attn_tc_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
        if (grid > 0)
            attn_tc_kernel<D, true><<<(unsigned)grid, kThreads, smem, st>>>(P, mq, mk, mv, A, ord);
    } else {
        const int smem = Layout<D, false>::kTotal;
        cudaFuncSetAttribute(attn_tc_kernel<D, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (grid > 0)
            attn_tc_kernel<D, false><<<(unsigned)grid, kThreads, smem, st>>>(P, mq, mk, mv, A, ord);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_partials(const DevProblem &P, const __nv_bfloat16 *q,
                                      const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                      const ScoreWs &ws, cudaStream_t s) {
    return P.d == 64 ? attention_d<64>(P, q, k, v, ws, s) : attention_d<128>(P, q, k, v, ws, s);
}

}  // namespace kvevict
