// kv_merge.cuh -- the split-K merge between the two streaming passes of the
// DropKV removal score, as a per-row device function (merge_row) that the
// stand-alone merge kernel (kv_score.cu) and the fused kernel (kv_fused.cu) call.
//
// Pass 1 leaves, for every unit, split of its keys (one or two partials per
// split) and window row (query head g of the GQA group, window slot t, causal
// position n - w + t), a partial (running max m in log2 units, sum l,
// unnormalised output o).  The merge combines them with the log-sum-exp rescale
// and stores, per row, (m, l), a = o / l split into a_hi = bf16(a) and
// a_lo = bf16(a - a_hi), and ||a_hi + a_lo||^2 -- the operands of the rescoring
// pass.  For the attention-sum rule the partials hold (m, l) only and the merge
// writes (m, l) alone (and ||a||^2 = 0).
#pragma once
#include <cfloat>

#include "kv_internal.cuh"

namespace kvevict {

// One warp merges window row `row` (< a_rows) of unit u; kO = false (the
// attention sum) merges (m, l) only.
template <int D, bool kO>
__device__ __forceinline__ void merge_row(const DevProblem &P, const ScoreWs &ws, long long u,
                                          int row, int lane) {
    if (!in_range((long long)u * ws.a_rows + row, P.units * ws.a_rows, ws.status)) return;
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
    const int nslots = (U.n + P.split_keys - 1) / P.split_keys * ws.parts;
    const size_t base = (size_t)u * P.max_splits * ws.parts * P.rows + row;
    // the unit's partial slots and its merged rows lie inside their arrays
    if (!in_range((long long)(base + (size_t)(nslots > 0 ? nslots - 1 : 0) * P.rows),
                  P.units * P.max_splits * ws.parts * P.rows, ws.status) ||
        !in_range((long long)u * P.rows + row, P.units * P.rows, ws.status) ||
        nslots > P.max_splits * ws.parts)
        return;

    // partials with l = 0 saw no key of this row (or no tile at all): skipped.
    // Lane j holds the (m, l) of slots j, j + 32, ...: loaded together.
    float M = -INFINITY;
    for (int s0 = 0; s0 < nslots; s0 += 32) {
        const int s = s0 + lane;
        const float2 ml = s < nslots ? ws.part_ml[base + (size_t)s * P.rows] : make_float2(0.f, 0.f);
        float m = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        M = fmaxf(M, m);
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
    // slots added in order; the o partials of four slots in flight at a time
    constexpr int kQ = 4;
    float Lsum = 0.f;
    for (int s0 = 0; s0 < nslots; s0 += 32) {
        const int cnt = min(32, nslots - s0);
        const float2 ml_l = lane < cnt ? ws.part_ml[base + (size_t)(s0 + lane) * P.rows]
                                       : make_float2(0.f, 0.f);
        const float f_l = ml_l.y > 0.f ? exp2f(ml_l.x - M) : 0.f;
        for (int j0 = 0; j0 < cnt; j0 += kQ) {
            float o[kQ][C];
            float fq[kQ], lq[kQ];
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                const int j = min(j0 + q, 31);
                fq[q] = __shfl_sync(0xffffffffu, f_l, j);
                lq[q] = __shfl_sync(0xffffffffu, ml_l.y, j);
                const bool use = j0 + q < cnt && lq[q] > 0.f;
                const float *po = ws.part_o + (base + (size_t)(s0 + j0 + q) * P.rows) * D;
#pragma unroll
                for (int i = 0; i < C; ++i) o[q][i] = use ? po[lane + 32 * i] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                if (j0 + q < cnt && lq[q] > 0.f) {
                    Lsum += lq[q] * fq[q];
#pragma unroll
                    for (int i = 0; i < C; ++i) a[i] += o[q][i] * fq[q];
                }
            }
        }
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

}  // namespace kvevict
