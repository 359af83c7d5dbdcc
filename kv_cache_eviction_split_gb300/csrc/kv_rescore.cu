// kv_rescore.cu -- pass 2 of the DropKV score on the tcgen05 tensor cores.
//
// For every key j of a unit and every window row r that sees it:
//     s   = q_r . k_j                         (tensor core, fp32 in TMEM)
//     X   = (a_hi_r + a_lo_r) . v_j           (tensor core, two bf16 MMAs)
//     e   = 2^(s * scale * log2 e - m_r)      p = e / l_r
//     x   = ||a_r||^2 - 2 X + ||v_j||^2      = ||a_r - v_j||^2 (the expansion the
//                                              DropKV scoring-kernel description uses)
//     S_j += e / (l_r - e) * sqrt(x)         = p/(1-p) * ||a_r - v_j||
// (DropKV, Key Contributions 1 and Methodology in Plain English).  a = a_hi +
// a_lo is the pass-1 output split into two bf16 halves, so the expansion keeps
// ~16 bits of a instead of bf16's 8.
//
// Orientation is key-major: one MMA tile is 128 keys (M, TMEM lanes) by the
// rows of a 128-row chunk of the unit's window rows (N), so each epilogue
// thread owns one key and sums its score over rows without any cross-thread
// reduction.  Work items = (unit, 64-key-tile block, row chunk); a persistent
// grid walks them round-robin, chunk fastest, so the chunks of one key block
// run on neighbouring SMs at the same time and share K/V through L2.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: the chunk's Q, a_hi, a_lo once per item; K and V
//               tiles through a 2-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread): per tile S = K Q^T and
//               X = V a_hi^T + V a_lo^T over all rows of the chunk, into one of
//               two TMEM buffers, so tile i+1 computes while tile i is scored
//               and a K/V stage frees as soon as its MMAs complete
//   warps 2-9   epilogue: group g (4 warps) handles half g of the rows; group 0
//               hands its per-key partial sums to group 1 through a smem ring
// Every wait is bounded: on expiry the kernel posts KV_ERR_TIMEOUT, the other
// roles drain out, TMEM is freed and the kernel returns.
#include <algorithm>
#include <cfloat>

#include "kv_internal.cuh"
#include "kv_sm100.cuh"

namespace kvevict {
namespace {
using namespace sm100;

constexpr int kTileKeys = 128;
constexpr int kChunkRows = 128;
constexpr int kTilesPerItem = 64;
constexpr int kStages = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kBlockBytes = kChunkRows * 128;   // one [128 rows][64 bf16] swizzled box

template <int D>
struct Layout {
    static constexpr int kOp = (D / 64) * kBlockBytes;     // one [128][D] bf16 operand
    static constexpr int kQ = 0;
    static constexpr int kAhi = kQ + kOp;
    static constexpr int kAlo = kAhi + kOp;
    static constexpr int kK = kAlo + kOp;
    static constexpr int kV = kK + kStages * kOp;
    static constexpr int kStats = kV + kStages * kOp;      // [2][32] float4 (-m0,-m1,l0,l1)
    static constexpr int kA2 = kStats + 2 * 32 * 16;       // [2][32] float2 ||a||^2 pairs
    static constexpr int kRmod = kA2 + 2 * 32 * 8;         // [2][64] uint16 row % w
    static constexpr int kRing = kRmod + 2 * 64 * 2;       // [2 slots][128] float
    static constexpr int kBars = kRing + 2 * 128 * 4;
    static constexpr int kNumBars = 4 * kStages + 2 + 8;
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kTotal = kMisc + 16;
};

struct RescoreArgs {
    const int32_t *plan;       // [units + 1] prefix of key-tile blocks per unit
    const float2 *stat_ml;     // [units][rows] (m in log2 units, l)
    const float *stat_a2;      // [units][rows]
    float *out;                // scores, or chunk partials [chunks][L*H*N_tot]
    long long out_stride;      // elements between chunk partials
    long long total_items;
    int chunks;
    int a_rows;                // rows per unit in a_hi / a_lo (chunks * 128)
    int *status;
};

struct Item {
    long long u;
    int c, t_begin, t_end;
};

__device__ __forceinline__ Item decode_item(long long item, const RescoreArgs &A, const DevProblem &P) {
    Item it;
    it.c = (int)(item % A.chunks);
    const long long gb = item / A.chunks;
    long long lo = 0, hi = P.units;            // plan[lo] <= gb < plan[hi]
    while (hi - lo > 1) {
        const long long mid = (lo + hi) >> 1;
        if (A.plan[mid] <= gb) lo = mid; else hi = mid;
    }
    it.u = lo;
    const int n = (int)(P.cu[(int)(lo / ((long long)P.L * P.H)) + 1] -
                        P.cu[(int)(lo / ((long long)P.L * P.H))]);
    const int tiles = (n + kTileKeys - 1) / kTileKeys;
    it.t_begin = (int)(gb - A.plan[lo]) * kTilesPerItem;
    it.t_end = min(it.t_begin + kTilesPerItem, tiles);
    return it;
}

__device__ __forceinline__ int chunk_half_rows(const DevProblem &P, int c) {
    const int rc = min(kChunkRows, P.rows - c * kChunkRows);
    return ((rc + 31) / 32) * 16;   // half of the chunk rows rounded up to 32
}

// ||v||^2 of one row of a swizzled [128][D] bf16 tile.
template <int D>
__device__ __forceinline__ float row_sqnorm(const uint8_t *tile, int row) {
    float acc = 0.f;
#pragma unroll
    for (int kb = 0; kb < D / 64; ++kb) {
        const uint8_t *base = tile + kb * kBlockBytes + row * 128;
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
            const uint4 w = *reinterpret_cast<const uint4 *>(base + ((c16 ^ (row & 7)) << 4));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(ws[i] << 16);
                const float hi = __uint_as_float(ws[i] & 0xFFFF0000u);
                acc = fmaf(lo, lo, acc);
                acc = fmaf(hi, hi, acc);
            }
        }
    }
    return acc;
}

// Adds the terms of 16 rows (columns of one TMEM load) for this thread's key:
// e/(l - e) * sqrt(x) with e = 2^(s c - m), x = max(||a||^2 - 2X + ||v||^2, 0),
// written as e * x * rsqrt((l - e)^2 x + tiny) so one MUFU op gives sqrt(x)/(l-e)
// and x = 0 gives 0.  Two rows at a time in packed f32x2 arithmetic.
__device__ __forceinline__ void rescore16(const float (&sv)[16], const float (&xv)[16],
                                          const float4 *st, const float2 *a2p,
                                          const uint16_t *rmod, bool boundary, int jrel,
                                          float cscale, float2 v2v2, float2 &acc) {
    const float2 cs2 = make_float2(cscale, cscale);
    const float2 neg1 = make_float2(-1.f, -1.f);
    const float2 neg2 = make_float2(-2.f, -2.f);
    const float2 tiny = make_float2(1e-30f, 1e-30f);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const float4 s4 = st[p];
        const float2 t = __ffma2_rn(make_float2(sv[2 * p], sv[2 * p + 1]), cs2,
                                    make_float2(s4.x, s4.y));
        const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        const float2 den = __ffma2_rn(e, neg1, make_float2(s4.z, s4.w));
        const float2 av = __fadd2_rn(a2p[p], v2v2);
        float2 x = __ffma2_rn(make_float2(xv[2 * p], xv[2 * p + 1]), neg2, av);
        x.x = fmaxf(x.x, 0.f);
        x.y = fmaxf(x.y, 0.f);
        const float2 y = __ffma2_rn(__fmul2_rn(den, den), x, tiny);
        float2 ex = __fmul2_rn(e, x);
        if (boundary) {
            if (jrel > (int)rmod[2 * p]) ex.x = 0.f;
            if (jrel > (int)rmod[2 * p + 1]) ex.y = 0.f;
        }
        acc = __ffma2_rn(ex, make_float2(rsqrt_approx(y.x), rsqrt_approx(y.y)), acc);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
rescore_tc_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ahi,
                  const __grid_constant__ CUtensorMap tm_alo, const RescoreArgs A) {
    using Ly = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly::kBars);
    uint64_t *k_full = bars, *k_empty = bars + kStages;
    uint64_t *v_full = bars + 2 * kStages, *v_empty = bars + 3 * kStages;
    uint64_t *qa_full = bars + 4 * kStages, *qa_empty = qa_full + 1;
    uint64_t *tm_full = qa_empty + 1, *tm_empty = tm_full + 2;
    uint64_t *part_full = tm_empty + 2, *part_empty = part_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Ly::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Ly::kMisc + 4);

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort_flag) post_status(A.status, KV_ERR_UNSUPPORTED);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1 + kEpiWarps);
        }
        mbar_init(qa_full, 1);
        mbar_init(qa_empty, 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&tm_full[h], 1);
            mbar_init(&tm_empty[h], kEpiWarps);
            mbar_init(&part_full[h], 4);
            mbar_init(&part_empty[h], 4);
        }
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_ahi);
        prefetch_tensormap(&tm_alo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool run = *abort_flag == 0;

    if (run && warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            long long tcount = 0, icount = 0;
            bool ok = true;
            for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
                const Item it = decode_item(item, A, P);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                ok = mbar_wait(qa_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, kWaitNs);
                if (!ok) break;
                mbar_arrive_expect_tx(qa_full, 3 * Ly::kOp);
                const int qy = (int)(U.q_row0 + it.c * kChunkRows);
                const int ay = (int)(it.u * A.a_rows + it.c * kChunkRows);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_load_2d(smem + Ly::kQ + kb * kBlockBytes, &tm_q, qa_full, kb * 64, qy);
                    tma_load_2d(smem + Ly::kAhi + kb * kBlockBytes, &tm_ahi, qa_full, kb * 64, ay);
                    tma_load_2d(smem + Ly::kAlo + kb * kBlockBytes, &tm_alo, qa_full, kb * 64, ay);
                }
                for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                    const int s = (int)(tcount % kStages);
                    const uint32_t par = (uint32_t)((tcount / kStages) & 1) ^ 1u;
                    const int ky = (int)(U.kv_row0 + (long long)t * kTileKeys);
                    ok = mbar_wait(&k_empty[s], par, abort_flag, kWaitNs);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&k_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kK + s * Ly::kOp + kb * kBlockBytes, &tm_k,
                                    &k_full[s], kb * 64, ky);
                    ok = mbar_wait(&v_empty[s], par, abort_flag, kWaitNs);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&v_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kV + s * Ly::kOp + kb * kBlockBytes, &tm_v,
                                    &v_full[s], kb * 64, ky);
                }
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            // drain: every load this thread issued lands before the CTA exits
            for (int s = 0; s < kStages; ++s) {
                const long long uses = tcount / kStages + ((tcount % kStages) > s ? 1 : 0);
                if (uses > 0) {
                    const uint32_t par = (uint32_t)((uses - 1) & 1);
                    mbar_wait(&k_full[s], par, abort_flag, kWaitNs);
                    mbar_wait(&v_full[s], par, abort_flag, kWaitNs);
                }
            }
        }
    } else if (run && warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            long long tcount = 0, icount = 0;
            bool ok = true;
            for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
                const Item it = decode_item(item, A, P);
                const int rch = chunk_half_rows(P, it.c);
                const uint32_t idesc = idesc_bf16_f32(128, 2 * rch);
                ok = mbar_wait(qa_full, (uint32_t)(icount & 1), abort_flag, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                const uint64_t qb = sdesc_k_sw128(smem_u32(smem + Ly::kQ));
                const uint64_t hb = sdesc_k_sw128(smem_u32(smem + Ly::kAhi));
                const uint64_t lb = sdesc_k_sw128(smem_u32(smem + Ly::kAlo));
                for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                    const int s = (int)(tcount % kStages);
                    const uint32_t par = (uint32_t)((tcount / kStages) & 1);
                    const int b = (int)(tcount & 1);          // TMEM buffer of this tile
                    ok = mbar_wait(&tm_empty[b], (uint32_t)((tcount >> 1) & 1) ^ 1u, abort_flag,
                                   kWaitNs) &&
                         mbar_wait(&k_full[s], par, abort_flag, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d_s = tmem + b * 256;
                    const uint32_t d_x = d_s + 128;
                    const uint64_t ka = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
                    const uint64_t va = sdesc_k_sw128(smem_u32(smem + Ly::kV + s * Ly::kOp));
                    mma_ss_c<false>(d_s, ka, qb, idesc);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            if (kb | kk)
                                mma_ss_c<true>(d_s, sdesc_add(ka, ko), sdesc_add(qb, ko), idesc);
                        }
                    mma_commit(&k_empty[s]);
                    ok = mbar_wait(&v_full[s], par, abort_flag, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    mma_ss_c<false>(d_x, va, hb, idesc);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            if (kb | kk)
                                mma_ss_c<true>(d_x, sdesc_add(va, ko), sdesc_add(hb, ko), idesc);
                        }
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            mma_ss_c<true>(d_x, sdesc_add(va, ko), sdesc_add(lb, ko), idesc);
                        }
                    mma_commit(&tm_full[b]);
                    mma_commit(&v_empty[s]);
                }
                mma_commit(qa_empty);
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
        }
    } else if (run) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int g = ew >> 2;                 // half of the chunk rows
        const int quarter = warp & 3;          // TMEM lane quarter this warp may access
        const int key_local = quarter * 32 + lane;
        const int tg = (ew & 3) * 32 + lane;   // thread index within the group
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float4 *stats = reinterpret_cast<float4 *>(smem + Ly::kStats) + g * 32;
        float2 *a2s = reinterpret_cast<float2 *>(smem + Ly::kA2) + g * 32;
        uint16_t *rmod = reinterpret_cast<uint16_t *>(smem + Ly::kRmod) + g * 64;
        float *ring = reinterpret_cast<float *>(smem + Ly::kRing);
        const float cscale = P.scale_log2;
        long long tcount = 0;
        bool ok = true;
        for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
            const Item it = decode_item(item, A, P);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int rch = chunk_half_rows(P, it.c);
            const int row_base = it.c * kChunkRows + g * rch;
            asm volatile("bar.sync %0, 128;" ::"r"(g + 1) : "memory");
            for (int pp = tg; pp < rch / 2; pp += 128) {
                float nm[2], ll[2], aa[2];
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    const int row = row_base + 2 * pp + k2;
                    if (row < P.rows) {
                        const float2 ml = A.stat_ml[it.u * P.rows + row];
                        nm[k2] = -ml.x;
                        ll[k2] = ml.y;
                        aa[k2] = A.stat_a2[it.u * P.rows + row];
                        rmod[2 * pp + k2] = (uint16_t)(row % P.w);
                    } else {   // padding row: e = 0, so its term is 0
                        nm[k2] = -INFINITY;
                        ll[k2] = 1.f;
                        aa[k2] = 0.f;
                        rmod[2 * pp + k2] = 0;
                    }
                }
                stats[pp] = make_float4(nm[0], nm[1], ll[0], ll[1]);
                a2s[pp] = make_float2(aa[0], aa[1]);
            }
            asm volatile("bar.sync %0, 128;" ::"r"(g + 1) : "memory");
            float *out = A.out + (long long)it.c * A.out_stride + U.kv_row0;
            const int pos0 = U.n - P.w;
            for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                const int s = (int)(tcount % kStages);
                const uint32_t spar = (uint32_t)((tcount / kStages) & 1);
                const int b = (int)(tcount & 1);              // TMEM buffer of this tile
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&tm_full[b], (uint32_t)((tcount >> 1) & 1), abort_flag,
                                          kWaitNs) &&
                                    mbar_wait(&v_full[s], spar, abort_flag, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                const float v2 = row_sqnorm<D>(smem + Ly::kV + s * Ly::kOp, key_local);
                __syncwarp();
                if (lane == 0) mbar_arrive(&v_empty[s]);
                const int j = t * kTileKeys + key_local;
                const bool boundary = t * kTileKeys + kTileKeys - 1 > pos0;
                // rows with j > pos0 + (row % w) do not see key j (only near the window)
                const int jrel = j - pos0;
                float2 acc = make_float2(0.f, 0.f);
                const float2 v2v2 = make_float2(v2, v2);
                const uint32_t s_col = tmem + lane_addr + b * 256 + g * rch;
                const uint32_t x_col = s_col + 128;
                float sA[16], xA[16], sB[16], xB[16];
                tmem_ld16(s_col, sA);
                tmem_ld16(x_col, xA);
                for (int cc = 0; cc < rch; cc += 32) {
                    tmem_ld_wait();
                    reg_fence(sA);
                    reg_fence(xA);
                    const bool second = cc + 16 < rch;
                    if (second) {
                        tmem_ld16(s_col + cc + 16, sB);
                        tmem_ld16(x_col + cc + 16, xB);
                    }
                    rescore16(sA, xA, stats + cc / 2, a2s + cc / 2, rmod + cc, boundary, jrel,
                              cscale, v2v2, acc);
                    if (second) {
                        tmem_ld_wait();
                        reg_fence(sB);
                        reg_fence(xB);
                        if (cc + 32 < rch) {
                            tmem_ld16(s_col + cc + 32, sA);
                            tmem_ld16(x_col + cc + 32, xA);
                        }
                        rescore16(sB, xB, stats + cc / 2 + 8, a2s + cc / 2 + 8, rmod + cc + 16,
                                  boundary, jrel, cscale, v2v2, acc);
                    }
                }
                const float acc_sum = acc.x + acc.y;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tm_empty[b]);
                const int slot = (int)(tcount & 1);
                const uint32_t rpar = (uint32_t)((tcount >> 1) & 1);
                if (g == 0) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&part_empty[slot], rpar ^ 1u, abort_flag, kWaitNs));
                    if (!ok) break;
                    ring[slot * 128 + key_local] = acc_sum;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&part_full[slot]);
                } else {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&part_full[slot], rpar, abort_flag, kWaitNs));
                    if (!ok) break;
                    const float tot = acc_sum + ring[slot * 128 + key_local];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&part_empty[slot]);
                    if (j < U.n) out[j] = tot;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            post_status(A.status, KV_ERR_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
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

template <int D>
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
    launch_plan(P, kTileKeys * kTilesPerItem, ws.plan, st);
    const long long blocks = total_blocks(P, kTileKeys * kTilesPerItem);
    const int chunks = ws.chunks;
    RescoreArgs A;
    A.plan = ws.plan;
    A.stat_ml = ws.stat_ml;
    A.stat_a2 = ws.stat_a2;
    A.out = chunks == 1 ? scores : ws.part_scores;
    A.out_stride = kv_rows;
    A.total_items = blocks * chunks;
    A.chunks = chunks;
    A.a_rows = ws.a_rows;
    A.status = ws.status;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = Layout<D>::kTotal;
    cudaFuncSetAttribute(rescore_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const long long grid = std::min<long long>(sms, A.total_items);
    if (grid > 0)
        rescore_tc_kernel<D><<<(unsigned)grid, kThreads, smem, st>>>(P, mq, mk, mv, mhi, mlo, A);
    if (chunks > 1)
        chunk_sum_kernel<<<sms * 8, 256, 0, st>>>(ws.part_scores, kv_rows, chunks, scores);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rescore(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, float *scores, const ScoreWs &ws,
                           cudaStream_t s) {
    return P.d == 64 ? rescore_d<64>(P, q, k, v, scores, ws, s)
                     : rescore_d<128>(P, q, k, v, scores, ws, s);
}

}  // namespace kvevict
