// kv_score.cu -- the two streaming passes of the DropKV removal score.
//
// Pass 1 (window attention, split-K): for every unit and every split of its
// keys, each window row (query head g of the GQA group, window slot t, causal
// position n - w + t) runs an online softmax over the split's keys and writes
// a partial (running max m in log2 units, sum l, unnormalised output o).  The
// merge combines the splits with the log-sum-exp rescale and stores, per row,
// (m, l), a = o / l split into a_hi = bf16(a) and a_lo = bf16(a - a_hi), and
// ||a_hi + a_lo||^2 -- the operands of the rescoring pass (kv_rescore.cu).
#include <cfloat>

#include "kv_internal.cuh"

namespace kvevict {
namespace {

constexpr int kP1Threads = 128;   // rows per pass-1 block
constexpr int kP1Keys = 32;       // keys per pass-1 tile

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

template <int D>
__global__ void __launch_bounds__(kP1Threads)
attn_partial_kernel(DevProblem P, const __nv_bfloat16 *__restrict__ q,
                    const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                    ScoreWs ws) {
    const int split = blockIdx.x;
    const long long u = blockIdx.y;
    const int chunk = blockIdx.z;
    const UnitInfo U = unit_info(P, u, P.cu);
    const int nsplit = (U.n + kSplitKeys - 1) / kSplitKeys;
    if (split >= nsplit) return;
    const int k_begin = split * kSplitKeys;
    const int k_end = min(U.n, k_begin + kSplitKeys);

    extern __shared__ float smem[];
    float *qT = smem;                     // [D][kP1Threads]
    float *Ks = qT + D * kP1Threads;      // [kP1Keys][D]
    float *Vs = Ks + kP1Keys * D;         // [kP1Keys][D]

    const int tid = threadIdx.x;
    const int row = chunk * kP1Threads + tid;
    const bool active = row < P.rows;
    const int pos = U.n - P.w + (row % P.w);

    for (int idx = tid; idx < kP1Threads * D; idx += kP1Threads) {
        const int rr = idx / D, c = idx % D;
        const int grow = chunk * kP1Threads + rr;
        qT[c * kP1Threads + rr] = grow < P.rows ? bf(q[(U.q_row0 + grow) * D + c]) : 0.f;
    }

    float o[D];
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int t0 = k_begin; t0 < k_end; t0 += kP1Keys) {
        __syncthreads();
        for (int idx = tid; idx < kP1Keys * D; idx += kP1Threads) {
            const int jj = idx / D, c = idx % D;
            const int key = t0 + jj;
            const bool ok = key < k_end;
            Ks[idx] = ok ? bf(k[(U.kv_row0 + key) * D + c]) : 0.f;
            Vs[idx] = ok ? bf(v[(U.kv_row0 + key) * D + c]) : 0.f;
        }
        __syncthreads();
        if (!active || t0 > pos) continue;

        float s[kP1Keys];
#pragma unroll
        for (int j = 0; j < kP1Keys; ++j) s[j] = 0.f;
        for (int c = 0; c < D; ++c) {
            const float qc = qT[c * kP1Threads + tid];
#pragma unroll
            for (int j = 0; j < kP1Keys; ++j) s[j] = fmaf(qc, Ks[j * D + c], s[j]);
        }
        float mt = m;
#pragma unroll
        for (int j = 0; j < kP1Keys; ++j) {
            const int key = t0 + j;
            s[j] = (key < k_end && key <= pos) ? s[j] * P.scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        const float corr = exp2f(m - mt);
        l *= corr;
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] *= corr;
#pragma unroll
        for (int j = 0; j < kP1Keys; ++j) {
            s[j] = exp2f(s[j] - mt);
            l += s[j];
        }
#pragma unroll
        for (int c = 0; c < D; ++c) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kP1Keys; ++j) acc = fmaf(s[j], Vs[j * D + c], acc);
            o[c] += acc;
        }
        m = mt;
    }
    if (!active) return;
    const size_t prow = ((size_t)u * P.max_splits + split) * P.rows + row;
    ws.part_ml[prow] = make_float2(m, l);
    float *po = ws.part_o + prow * D;
#pragma unroll
    for (int c = 0; c < D; ++c) po[c] = o[c];
}

template <int D>
__global__ void __launch_bounds__(128)
attn_merge_kernel(DevProblem P, ScoreWs ws) {
    const long long u = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.y * 4 + warp;
    if (row >= ws.a_rows) return;
    if (row >= P.rows) {   // padding rows of the last 128-row chunk read as zeros
        const size_t arow = (size_t)u * ws.a_rows + row;
        for (int c = lane; c < D; c += 32) {
            ws.a_hi[arow * D + c] = __float2bfloat16_rn(0.f);
            ws.a_lo[arow * D + c] = __float2bfloat16_rn(0.f);
        }
        return;
    }
    const UnitInfo U = unit_info(P, u, P.cu);
    const int nsplit = (U.n + kSplitKeys - 1) / kSplitKeys;
    const size_t base = (size_t)u * P.max_splits * P.rows + row;

    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ws.part_ml[base + (size_t)s * P.rows].x);
    constexpr int C = D / 32;
    float a[C];
#pragma unroll
    for (int i = 0; i < C; ++i) a[i] = 0.f;
    float Lsum = 0.f;
    for (int s = 0; s < nsplit; ++s) {
        const size_t pr = base + (size_t)s * P.rows;
        const float2 ml = ws.part_ml[pr];
        const float f = exp2f(ml.x - M);
        Lsum += ml.y * f;
        const float *po = ws.part_o + pr * D;
#pragma unroll
        for (int i = 0; i < C; ++i) a[i] += po[lane + 32 * i] * f;
    }
    const float inv = 1.f / Lsum;
    float a2 = 0.f;
    const size_t srow = (size_t)u * P.rows + row;
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

template <typename K>
void set_smem(K kernel, size_t bytes) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D>
cudaError_t attention_d(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                        const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t st) {
    const size_t smem = sizeof(float) * (D * kP1Threads + 2 * kP1Keys * D);
    set_smem(attn_partial_kernel<D>, smem);
    dim3 g1(P.max_splits, (unsigned)P.units, (P.rows + kP1Threads - 1) / kP1Threads);
    attn_partial_kernel<D><<<g1, kP1Threads, smem, st>>>(P, q, k, v, ws);
    dim3 g2((unsigned)P.units, (ws.a_rows + 3) / 4);
    attn_merge_kernel<D><<<g2, 128, 0, st>>>(P, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t s) {
    return P.d == 64 ? attention_d<64>(P, q, k, v, ws, s) : attention_d<128>(P, q, k, v, ws, s);
}

}  // namespace kvevict
