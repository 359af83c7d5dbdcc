// kv_rescore.cu -- the stand-alone pass-2 kernel (body in kv_pass2.cuh), the
// sum of the row-chunk partials, and their launcher.
#include <algorithm>

#include "kv_pass2.cuh"

namespace kvevict {
namespace {
using namespace sm100;
using namespace pass2;

template <int D, int RULE>
__global__ void __launch_bounds__(kThreads, 1)
rescore_tc_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ahi,
                  const __grid_constant__ CUtensorMap tm_alo, const RescoreArgs A,
                  const __grid_constant__ ItemOrder ord) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t tmem =
        tmem_acquire_all(reinterpret_cast<uint32_t *>(smem + Layout<D, RULE>::kMisc));
    rescore_body<D, RULE>(P, &tm_q, &tm_k, &tm_v, &tm_ahi, &tm_alo, A, ord, smem, tmem, blockIdx.x,
                          gridDim.x);
    tmem_release_all(tmem);
}

// scores = sum over chunks of the chunk partials, in chunk order.
__global__ void chunk_sum_kernel(const float *__restrict__ part, long long stride, int chunks,
                                 float *__restrict__ out) {
    const long long step = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < stride; i += step) {
        float acc = part[i];
        for (int c = 1; c < chunks; ++c) acc += part[c * stride + i];
        out[i] = acc;
    }
}

template <int D, int RULE>
cudaError_t rescore_d(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                      const __nv_bfloat16 *v, float *scores, const ScoreWs &ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mhi, mlo;
    const long long q_rows = (long long)P.R * P.L * P.Hq * P.w;
    const long long kv_rows = (long long)P.L * P.H * P.N_tot;
    const long long a_rows = P.units * ws.a_rows;
    if (!make_tile_map(&mq, q, q_rows, D) || !make_tile_map(&mk, k, kv_rows, D) ||
        !make_tile_map(&mv, v, kv_rows, D) || !make_tile_map(&mhi, ws.a_hi, a_rows, D) ||
        !make_tile_map(&mlo, ws.a_lo, a_rows, D))
        return cudaErrorInvalidValue;
    ItemOrder ord;
    build_item_order(P, kPass2BlockKeys, &ord);
    if (ord.nrun == 0)   // only with more runs of lengths than the order tables hold
        launch_plan(P, kTileKeys * kTilesPerItem, ws.plan, st);
    const long long blocks = total_blocks(P, kTileKeys * kTilesPerItem);
    const int chunks = ws.chunks;
    RescoreArgs A;
    A.plan = ws.plan;
    A.stat_ml = ws.stat_ml;
    A.stat_a2 = ws.stat_a2;
    A.v2 = ws.v2;
    A.out = chunks == 1 ? scores : ws.part_scores;
    A.out_stride = kv_rows;
    A.total_items = blocks * chunks;
    A.chunks = chunks;
    A.a_rows = ws.a_rows;
    A.status = ws.status;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = Layout<D, RULE>::kTotal;
    cudaFuncSetAttribute(rescore_tc_kernel<D, RULE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         smem);
    const long long grid = std::min<long long>(sms, A.total_items);
    if (grid > 0)
        rescore_tc_kernel<D, RULE>
            <<<(unsigned)grid, kThreads, smem, st>>>(P, mq, mk, mv, mhi, mlo, A, ord);
    if (chunks > 1)
        chunk_sum_kernel<<<sms * 8, 256, 0, st>>>(ws.part_scores, kv_rows, chunks, scores);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rescore(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, float *scores, const ScoreWs &ws,
                           cudaStream_t s) {
    switch (P.rule) {
        case KV_SCORE_DROPKV_SQUARED:
            return P.d == 64 ? rescore_d<64, KV_SCORE_DROPKV_SQUARED>(P, q, k, v, scores, ws, s)
                             : rescore_d<128, KV_SCORE_DROPKV_SQUARED>(P, q, k, v, scores, ws, s);
        case KV_SCORE_ATTN_SUM:
            return P.d == 64 ? rescore_d<64, KV_SCORE_ATTN_SUM>(P, q, k, v, scores, ws, s)
                             : rescore_d<128, KV_SCORE_ATTN_SUM>(P, q, k, v, scores, ws, s);
        default:
            return P.d == 64 ? rescore_d<64, KV_SCORE_DROPKV>(P, q, k, v, scores, ws, s)
                             : rescore_d<128, KV_SCORE_DROPKV>(P, q, k, v, scores, ws, s);
    }
}

}  // namespace kvevict
