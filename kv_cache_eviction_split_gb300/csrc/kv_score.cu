// kv_score.cu -- the split-K merge between the two streaming passes of the
// DropKV removal score.
//
// Pass 1 (kv_attention.cu) leaves, for every unit, split of its keys (one or two
// partials per split) and window row (query head g of the GQA group, window slot
// t, causal position n - w + t), a partial (running max m in log2 units, sum l,
// unnormalised output o).  The merge combines them with the log-sum-exp rescale
// and stores, per row,
// (m, l), a = o / l split into a_hi = bf16(a) and a_lo = bf16(a - a_hi), and
// ||a_hi + a_lo||^2 -- the operands of the rescoring pass (kv_rescore.cu).  For
// the attention-sum rule the partials hold (m, l) only and the merge writes
// (m, l) alone (and ||a||^2 = 0).
#include <cfloat>

#include "kv_internal.cuh"

namespace kvevict {
namespace {

template <int D, bool kO>
__global__ void __launch_bounds__(128)
attn_merge_kernel(DevProblem P, ScoreWs ws) {
    const long long u = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.y * 4 + warp;
    if (row >= ws.a_rows) return;
    if (kO && row >= P.rows) {   // padding rows of the last 128-row chunk read as zeros
        const size_t arow = (size_t)u * ws.a_rows + row;
        for (int c = lane; c < D; c += 32) {
            ws.a_hi[arow * D + c] = __float2bfloat16_rn(0.f);
            ws.a_lo[arow * D + c] = __float2bfloat16_rn(0.f);
        }
        return;
    }
    if (!kO && row >= P.rows) return;
    const UnitInfo U = unit_info(P, u, P.cu);
    const int nslots = (U.n + kSplitKeys - 1) / kSplitKeys * ws.parts;
    const size_t base = (size_t)u * P.max_splits * ws.parts * P.rows + row;

    // partials with l = 0 saw no key of this row (or no tile at all): skipped
    float M = -INFINITY;
    for (int s = 0; s < nslots; ++s) {
        const float2 ml = ws.part_ml[base + (size_t)s * P.rows];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    const size_t srow = (size_t)u * P.rows + row;
    if constexpr (!kO) {
        float Lsum = 0.f;
        for (int s = lane; s < nslots; s += 32) {
            const float2 ml = ws.part_ml[base + (size_t)s * P.rows];
            if (ml.y > 0.f) Lsum += ml.y * exp2f(ml.x - M);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
        if (lane == 0) {
            ws.stat_ml[srow] = make_float2(M, Lsum);
            ws.stat_a2[srow] = 0.f;
        }
        return;
    }
    constexpr int C = D / 32;
    float a[C];
#pragma unroll
    for (int i = 0; i < C; ++i) a[i] = 0.f;
    float Lsum = 0.f;
    for (int s = 0; s < nslots; ++s) {
        const size_t pr = base + (size_t)s * P.rows;
        const float2 ml = ws.part_ml[pr];
        if (!(ml.y > 0.f)) continue;
        const float f = exp2f(ml.x - M);
        Lsum += ml.y * f;
        const float *po = ws.part_o + pr * D;
#pragma unroll
        for (int i = 0; i < C; ++i) a[i] += po[lane + 32 * i] * f;
    }
    const float inv = 1.f / Lsum;
    float a2 = 0.f;
    const size_t arow = (size_t)u * ws.a_rows + row;
#pragma unroll
    for (int i = 0; i < C; ++i) {
        const float av = a[i] * inv;
        const __nv_bfloat16 hi = __float2bfloat16_rn(av);
        const __nv_bfloat16 lo = __float2bfloat16_rn(av - __bfloat162float(hi));
        ws.a_hi[arow * D + lane + 32 * i] = hi;
        ws.a_lo[arow * D + lane + 32 * i] = lo;
        const float sum = __bfloat162float(hi) + __bfloat162float(lo);
        a2 = fmaf(sum, sum, a2);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a2 += __shfl_xor_sync(0xffffffffu, a2, off);
    if (lane == 0) {
        ws.stat_ml[srow] = make_float2(M, Lsum);
        ws.stat_a2[srow] = a2;
    }
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
