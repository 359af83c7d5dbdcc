// kv_fused.cu -- the whole eviction path in one launch.
//
// One persistent cooperative kernel (one 384-thread CTA per SM, all resident at
// once) runs the path's steps as phases, separated by grid-wide barriers:
//   0. the work plans of both passes (prefix sums of key blocks per unit)
//   1. pass 1: split-K window attention partials (row statistics alone for the
//      attention sum)                                         -- kv_pass1.cuh
//   2. the split merge: (m, l), a_hi, a_lo, ||a||^2 per row   -- kv_merge.cuh
//   3. pass 2: the per-key scores                             -- kv_pass2.cuh
//   4. the sum of the row-chunk partials (when rows span several chunks)
//   5. the budgeted top-k of every unit                      -- kv_select.cuh
//   6. the compaction of the kept K/V rows                    -- kv_compact.cuh
// The phases run the same device code as the stand-alone kernels, so the
// results are bit-identical to kv_score + kv_select_topk + kv_compact.  What
// the fusion removes is the host's part: eight launches and the gaps between
// them become one launch.
//
// Each barrier is a counter in the score workspace header (zeroed by an
// in-stream memset before the launch): a CTA adds one on arrival and waits,
// bounded by the pipeline wait limit, until all CTAs of the phase have arrived.
// A CTA whose wait expires posts KV_ERR_TIMEOUT and sets the abort word, which
// the other CTAs' waits watch; from then on every CTA skips the remaining
// phases (still passing each barrier, which then returns at once) and exits.
// Data one phase writes and a later phase reads is read with coherent loads
// (never the read-only path), and generic-proxy global writes are fenced
// against the TMA reads of the next phase at every barrier.
#include <algorithm>

#include "kv_compact.cuh"
#include "kv_merge.cuh"
#include "kv_pass1.cuh"
#include "kv_pass2.cuh"
#include "kv_select.cuh"

namespace kvevict {
namespace {
using namespace sm100;

constexpr int kFusedThreads = 384;     // pass 1's warp roles; pass 2 leaves two warps idle
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedCompactUnroll = 8;  // one CTA per SM: more rows in flight per warp
constexpr long long kFusedCompactRows = 2048;   // output rows per compaction item
constexpr int kFusedSelLoads = 16;      // keys in flight per thread in the radix passes
constexpr int kFusedSelItems = 16;      // candidates per thread per ordered-pass round

struct FusedArgs {
    pass1::AttnArgs a1;
    pass2::RescoreArgs a2;
    ScoreWs ws;
    float *scores;
    const int32_t *budgets;
    const int64_t *offsets;
    int32_t *sel;
    const uint4 *k16, *v16;     // K, V as 16-byte chunks (compaction)
    uint4 *kout, *vout;
    long long total_rows;
    unsigned *bar;              // [0] arrivals, [16] abort word
};

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int RULE>
struct FusedSmem {
    static constexpr int kP1 = RULE == KV_SCORE_ATTN_SUM
                                   ? pass1::StatLayout<D>::kTotal
                                   : cmax(pass1::Layout<D, false>::kTotal,
                                          pass1::Layout<D, true>::kTotal);
    static constexpr int kP2 = pass2::Layout<D, RULE>::kTotal;
    static constexpr int kSel = sel_smem_bytes<kFusedThreads, kFusedSelItems>();
    static constexpr int kSlot = (cmax(cmax(kP1, kP2), kSel) + 15) / 16 * 16;
    // the TMEM base slot last; at least 118 KB, more than half of an SM's 228 KB,
    // so no two CTAs share an SM (each holds all 512 TMEM columns, and one waiting
    // to allocate would stall the grid barriers)
    static constexpr int kTotal = cmax(kSlot + 16, 118 * 1024);
};

// plan[u] = sum over units u' < u of ceil(n_u' / keys_per_block); plan[units]
// = total.  One warp, 32 units a step.
__device__ __forceinline__ void plan_warp(const DevProblem &P, int keys_per_block, int32_t *plan) {
    const int lane = threadIdx.x & 31;
    int32_t run = 0;
    for (long long u0 = 0; u0 < P.units; u0 += 32) {
        const long long u = u0 + lane;
        int32_t b = 0;
        if (u < P.units) {
            const int r = (int)(u / ((long long)P.L * P.H));
            const int n = (int)(P.cu[r + 1] - P.cu[r]);
            b = (n + keys_per_block - 1) / keys_per_block;
        }
        int32_t incl = b;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (u < P.units) plan[u] = run + incl - b;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) plan[P.units] = run;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number target / gridDim.x.  Returns false in every thread of
// the CTA if the barrier was aborted or this CTA's wait expired.
__device__ __forceinline__ bool grid_sync(unsigned *bar, unsigned target, int *status,
                                          unsigned long long wait_ns) {
    fence_proxy_async_global();
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(bar, 1u);
        const unsigned long long t0 = globaltimer_ns();
        while (ld_acquire_gpu(bar) < target) {
            if (ld_acquire_gpu(bar + 16) != 0u) {
                ok = 0;
                break;
            }
            if (globaltimer_ns() - t0 > wait_ns) {
                atomicExch(bar + 16, 1u);
                post_status(status, KV_ERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(256);
        }
        __threadfence();
    }
    ok = __syncthreads_and(ok);
    fence_proxy_async_global();
    return ok != 0;
}

// scores = sum of the row-chunk partials in chunk order; 16-byte vectors, four
// in flight per thread, when the partials' stride allows them.
__device__ __forceinline__ void chunk_sum_phase(const FusedArgs &F, long long cta,
                                                long long ncta) {
    const long long stride = F.a2.out_stride;
    const int chunks = F.ws.chunks;
    const float *part = F.ws.part_scores;
    const long long t0 = cta * kFusedThreads + threadIdx.x, step = ncta * kFusedThreads;
    if ((stride & 3) == 0) {
        constexpr int kU = 4;
        const long long n4 = stride >> 2;
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        float4 *o4 = reinterpret_cast<float4 *>(F.scores);
        for (long long i0 = t0; i0 < n4; i0 += step * kU) {
            float4 acc[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const long long i = i0 + q * step;
                if (i < n4) acc[q] = p4[i];
            }
            for (int c = 1; c < chunks; ++c) {
#pragma unroll
                for (int q = 0; q < kU; ++q) {
                    const long long i = i0 + q * step;
                    if (i < n4) {
                        const float4 x = p4[(long long)c * n4 + i];
                        acc[q].x += x.x;
                        acc[q].y += x.y;
                        acc[q].z += x.z;
                        acc[q].w += x.w;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const long long i = i0 + q * step;
                if (i < n4) o4[i] = acc[q];
            }
        }
    } else {
        for (long long i = t0; i < stride; i += step) {
            float acc = part[i];
            for (int c = 1; c < chunks; ++c) acc += part[c * stride + i];
            F.scores[i] = acc;
        }
    }
}

template <int D, int RULE>
__global__ void __launch_bounds__(kFusedThreads, 1)
fused_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const __grid_constant__ CUtensorMap tm_ahi,
             const __grid_constant__ CUtensorMap tm_alo, const FusedArgs F,
             const __grid_constant__ ItemOrder ord1, const __grid_constant__ ItemOrder ord2) {
    using Sm = FusedSmem<D, RULE>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const long long cta = blockIdx.x, ncta = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t tmem = tmem_acquire_all(reinterpret_cast<uint32_t *>(smem + Sm::kSlot));
    unsigned phase = 0;
    auto barrier = [&]() {
        ++phase;
        return grid_sync(F.bar, phase * (unsigned)ncta, F.ws.status, P.wait_ns);
    };

    // 0. work plans
    if (cta == 0 && warp < 2)
        plan_warp(P, warp == 0 ? P.split_keys : pass2::kTileKeys * pass2::kTilesPerItem,
                  warp == 0 ? F.ws.plan : F.ws.plan2);
    bool ok = barrier();
    // 1. pass 1
    if (ok) {
        if constexpr (RULE == KV_SCORE_ATTN_SUM)
            pass1::attn_stats_body<D>(P, &tm_q, &tm_k, F.a1, ord1, smem, tmem, cta, ncta);
        else if (F.a1.parts == 2)   // one row chunk: one Q slot, a third V stage
            pass1::attn_tc_body<D, true>(P, &tm_q, &tm_k, &tm_v, F.a1, ord1, smem, tmem, cta,
                                         ncta);
        else
            pass1::attn_tc_body<D, false>(P, &tm_q, &tm_k, &tm_v, F.a1, ord1, smem, tmem, cta,
                                          ncta);
    }
    ok = barrier() && ok;
    // 2. merge: one warp per (unit, row)
    if (ok) {
        const long long rows_total = P.units * F.ws.a_rows;
        for (long long g = cta * kFusedWarps + warp; g < rows_total; g += ncta * kFusedWarps)
            merge_row<D, RULE != KV_SCORE_ATTN_SUM>(P, F.ws, g / F.ws.a_rows,
                                                    (int)(g % F.ws.a_rows), lane);
    }
    ok = barrier() && ok;
    // 3. pass 2
    if (ok)
        pass2::rescore_body<D, RULE, true>(P, &tm_q, &tm_k, &tm_v, &tm_ahi, &tm_alo, F.a2, ord2,
                                           smem, tmem, cta, ncta);
    ok = barrier() && ok;
    // 4. chunk partials -> scores, in chunk order
    if (F.ws.chunks > 1) {
        if (ok) chunk_sum_phase(F, cta, ncta);
        ok = barrier() && ok;
    }
    // 5. top-k: units round-robin over the CTAs
    if (ok) {
        const SelSmem sm = sel_smem<kFusedThreads>(smem);   // chunk_keys sized for kFusedSelItems
        for (long long u = cta; u < P.units; u += ncta) {
            __syncthreads();
            select_unit<kFusedThreads, true, kFusedSelLoads, kFusedSelItems>(
                P, F.scores, F.budgets, F.offsets, F.sel, F.ws.status, u, sm);
        }
    }
    ok = barrier() && ok;
    // 6. compaction: ranges of output rows round-robin over the CTAs
    if (ok && F.total_rows > 0) {
        const long long items = (F.total_rows + kFusedCompactRows - 1) / kFusedCompactRows;
        for (long long it = cta; it < items; it += ncta) {
            const long long r0 = it * kFusedCompactRows;
            compact_rows<D, kFusedWarps, kFusedCompactUnroll>(
                P, F.k16, F.v16, F.sel, F.offsets, r0,
                std::min(F.total_rows, r0 + kFusedCompactRows), F.kout, F.vout);
        }
    }
    tc_fence_before();
    __syncthreads();
    tmem_release_all(tmem);
}

template <int D, int RULE>
cudaError_t fused_d(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                    const __nv_bfloat16 *v, const int32_t *budgets, const int64_t *offsets,
                    long long total_rows, float *scores, int32_t *sel, __nv_bfloat16 *kout,
                    __nv_bfloat16 *vout, const ScoreWs &ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv, mhi, mlo;
    const long long q_rows = (long long)P.R * P.L * P.Hq * P.w;
    const long long kv_rows = (long long)P.L * P.H * P.N_tot;
    const long long a_rows = P.units * ws.a_rows;
    if (!make_tile_map(&mq, q, q_rows, D) || !make_tile_map(&mk, k, kv_rows, D) ||
        !make_tile_map(&mv, v, kv_rows, D) || !make_tile_map(&mhi, ws.a_hi, a_rows, D) ||
        !make_tile_map(&mlo, ws.a_lo, a_rows, D))
        return cudaErrorInvalidValue;
    FusedArgs F{};
    ItemOrder ord1, ord2;                // kernel parameters: the item decode reads them in place
    build_item_order(P, P.split_keys, &ord1);
    build_item_order(P, kPass2BlockKeys, &ord2);
    F.a1.plan = ws.plan;
    F.a1.part_ml = ws.part_ml;
    F.a1.part_o = ws.part_o;
    F.a1.v2 = ws.v2;
    F.a1.chunks = ws.chunks;
    F.a1.parts = ws.parts;
    F.a1.pairs = ws.parts == 1 ? (ws.chunks + 1) / 2 : 1;
    F.a1.total_items = total_blocks(P, P.split_keys) * F.a1.pairs;
    F.a1.status = ws.status;
    F.a2.plan = ws.plan2;
    F.a2.stat_ml = ws.stat_ml;
    F.a2.stat_a2 = ws.stat_a2;
    F.a2.v2 = ws.v2;
    F.a2.out = ws.chunks == 1 ? scores : ws.part_scores;
    F.a2.out_stride = kv_rows;
    F.a2.total_items =
        total_blocks(P, pass2::kTileKeys * pass2::kTilesPerItem) * (long long)ws.chunks;
    F.a2.chunks = ws.chunks;
    F.a2.a_rows = ws.a_rows;
    F.a2.status = ws.status;
    F.ws = ws;
    F.scores = scores;
    F.budgets = budgets;
    F.offsets = offsets;
    F.sel = sel;
    F.k16 = reinterpret_cast<const uint4 *>(k);
    F.v16 = reinterpret_cast<const uint4 *>(v);
    F.kout = reinterpret_cast<uint4 *>(kout);
    F.vout = reinterpret_cast<uint4 *>(vout);
    F.total_rows = total_rows;
    F.bar = reinterpret_cast<unsigned *>(reinterpret_cast<char *>(ws.status) + kGridBarOffset);
    // the whole header: the status word (a new sequence) and the barrier words
    cudaError_t e = cudaMemsetAsync(ws.status, 0, kHeaderBytes, st);
    if (e != cudaSuccess) return e;

    auto kern = fused_kernel<D, RULE>;
    const int smem = FusedSmem<D, RULE>::kTotal;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, smem);
    if (e != cudaSuccess) return e;
    if (!coop || per_sm != 1) return cudaErrorCooperativeLaunchTooLarge;
    DevProblem Pc = P;
    void *args[] = {&Pc, &mq, &mk, &mv, &mhi, &mlo, &F, &ord1, &ord2};
    // one CTA per SM: each holds all 512 TMEM columns
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(kern), dim3((unsigned)sms),
                                       dim3(kFusedThreads), args, (size_t)smem, st);
}

template <int D>
cudaError_t fused_rule(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                       const __nv_bfloat16 *v, const int32_t *budgets, const int64_t *offsets,
                       long long total_rows, float *scores, int32_t *sel, __nv_bfloat16 *kout,
                       __nv_bfloat16 *vout, const ScoreWs &ws, cudaStream_t s) {
    switch (P.rule) {
        case KV_SCORE_DROPKV_SQUARED:
            return fused_d<D, KV_SCORE_DROPKV_SQUARED>(P, q, k, v, budgets, offsets, total_rows,
                                                       scores, sel, kout, vout, ws, s);
        case KV_SCORE_ATTN_SUM:
            return fused_d<D, KV_SCORE_ATTN_SUM>(P, q, k, v, budgets, offsets, total_rows, scores,
                                                 sel, kout, vout, ws, s);
        default:
            return fused_d<D, KV_SCORE_DROPKV>(P, q, k, v, budgets, offsets, total_rows, scores,
                                               sel, kout, vout, ws, s);
    }
}

}  // namespace

cudaError_t launch_fused(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                         const __nv_bfloat16 *v, const int32_t *budgets, const int64_t *offsets,
                         long long total_rows, float *scores, int32_t *sel, __nv_bfloat16 *kout,
                         __nv_bfloat16 *vout, const ScoreWs &ws, cudaStream_t s) {
    return P.d == 64 ? fused_rule<64>(P, q, k, v, budgets, offsets, total_rows, scores, sel, kout,
                                      vout, ws, s)
                     : fused_rule<128>(P, q, k, v, budgets, offsets, total_rows, scores, sel,
                                       kout, vout, ws, s);
}

}  // namespace kvevict
