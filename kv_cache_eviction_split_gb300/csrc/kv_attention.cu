// kv_attention.cu -- pass 1 of the DropKV score on the tcgen05 tensor cores:
// causal window attention over each unit's keys, split across CTAs (split-K),
// producing per split the row max m (log2 units), the row sum l of
// 2^(s*scale*log2 e - m) and the unnormalised output O = sum_j P_j v_j.  The
// merge in kv_score.cu combines the splits (DropKV, "Methodology in Plain
// English": the attention output a whose removal shift the score measures).
//
// Query-major, one 128-row chunk of the unit's G*w window rows per work item:
//   S = Q K^T    M = 128 rows, N = 128 keys, K = d   (fp32 in TMEM, 3 buffers)
//   O += P V     M = 128 rows, N = d, K = 128 keys   (fp32 in TMEM; P is the
//                A operand read from TMEM, V the MN-major B operand in smem)
// The softmax warps turn S into P = 2^(s c - m) and store it, as two bf16
// halves P_hi = bf16(p) and P_lo = bf16(p - P_hi), back into the TMEM columns
// of the same S buffer (each 16-key chunk's 16 columns hold its 8 P_hi then 8
// P_lo columns); O accumulates P_hi V + P_lo V.  (A single bf16 P
// leaves a with ~2^-9 relative error, which the rescoring expansion amplifies
// where a is close to a value row; the split keeps ~16 bits of p.)  Because P
// lives in the S buffer, P is triple-buffered with S: S of tile i+1 and the
// softmax of tile i+1 overlap P V of tile i.
//
// Softmax details: tile max with the causal mask; a lazy rescale (O and l are
// rescaled only when the tile max exceeds the running max by more than 2^8,
// so every exponent stays <= 2^8); row sums from the unrounded fp32 p.  Warps
// w and w+4 share the 32 rows of TMEM lane quarter w % 4, each taking 64 of a
// tile's 128 keys and half of O's columns; they agree on the row max through
// shared memory.
//
// Barrier parities are tracked from use counts; no barrier can run more than
// one phase ahead of its waiter (the S/P buffer of tile i is only refilled
// after P V of tile i-3 completes).
//
// Warp roles (320 threads): warp 0 TMA producer (Q chunk per item, K and V
// tiles through a 3-stage ring); warp 1 TMEM owner and MMA issuer, running
// S of tile i+1 ahead of P V of tile i; warps 2-9 softmax.  Work items are
// (unit, 16384-key split, row chunk), chunk fastest, walked round-robin by a
// persistent grid.  All waits are bounded (KV_ERR_TIMEOUT on expiry).
#include <cfloat>

#include "kv_internal.cuh"
#include "kv_sm100.cuh"

namespace kvevict {
namespace {
using namespace sm100;

constexpr int kTileKeys = 128;
constexpr int kChunkRows = 128;
constexpr int kStages = 3;
constexpr int kPrefetchTiles = 4;   // K/V tiles requested into L2 ahead of the smem loads
constexpr int kSoftWarps = 8;
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                    // S/P buffers in TMEM
constexpr uint32_t kOCol = kSBufs * 128;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kBlockBytes = 128 * 128;       // [128 rows][64 bf16], 128 B swizzle
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct Layout {
    static constexpr int kOp = (D / 64) * kBlockBytes;   // [128][D] bf16
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kOp;
    static constexpr int kV = kK + kStages * kOp;
    static constexpr int kXmax = kV + kStages * kOp;      // [2 slots][2 halves][128] float
    static constexpr int kXl = kXmax + 2 * 2 * 128 * 4;    // [128] float
    static constexpr int kBars = kXl + 128 * 4;
    static constexpr int kNumBars = 4 * kStages + 2 + 3 * kSBufs + 2 + 8 + 4;
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kTotal = kMisc + 16;
};

struct AttnArgs {
    const int32_t *plan;       // [units + 1] prefix of key splits per unit
    float2 *part_ml;           // [units][max_splits][rows]
    float *part_o;             // [units][max_splits][rows][d]
    long long total_items;
    int chunks;
    int *status;
};

struct Item {
    long long u;
    int c, split, t0, t1;
};

__device__ __forceinline__ Item decode_item(long long item, const AttnArgs &A, const DevProblem &P) {
    Item it;
    it.c = (int)(item % A.chunks);
    const long long gs = item / A.chunks;
    long long lo = 0, hi = P.units;
    while (hi - lo > 1) {
        const long long mid = (lo + hi) >> 1;
        if (A.plan[mid] <= gs) lo = mid; else hi = mid;
    }
    it.u = lo;
    const int r = (int)(lo / ((long long)P.L * P.H));
    const int n = (int)(P.cu[r + 1] - P.cu[r]);
    it.split = (int)(gs - A.plan[lo]);
    const int k0 = it.split * kSplitKeys;
    const int k1 = min(n, k0 + kSplitKeys);
    it.t0 = k0 / kTileKeys;
    it.t1 = (k1 + kTileKeys - 1) / kTileKeys;
    return it;
}

// p = 2^(s c - m) for 16 keys held in registers; adds p to the row sum and
// stores bf16(p) at TMEM column hi_col and bf16(p - bf16(p)) at lo_col (8
// columns each, two keys per column, the lower key in the low half).
template <bool kMasked>
__device__ __forceinline__ void soft16_tmem(const float *v, int j0, int lim, float cs,
                                            float negm, float2 &lsum, uint32_t hi_col,
                                            uint32_t lo_col) {
    const float2 cs2 = make_float2(cs, cs);
    const float2 nm2 = make_float2(negm, negm);
    const float2 neg1 = make_float2(-1.f, -1.f);
    uint32_t whi[8], wlo[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        const int j = 2 * h;
        const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), cs2, nm2);
        float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        if (kMasked) {
            if (j0 + j > lim) p.x = 0.f;
            if (j0 + j + 1 > lim) p.y = 0.f;
        }
        lsum = __fadd2_rn(lsum, p);
        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(p.x, p.y);
        const float2 lo = __ffma2_rn(__bfloat1622float2(hi2), neg1, p);
        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(lo.x, lo.y);
        whi[h] = *reinterpret_cast<const uint32_t *>(&hi2);
        wlo[h] = *reinterpret_cast<const uint32_t *>(&lo2);
    }
    tmem_st8u(hi_col, whi);
    tmem_st8u(lo_col, wlo);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const DevProblem P, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const AttnArgs A) {
    using Ly = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly::kBars);
    uint64_t *k_full = bars, *k_empty = bars + kStages;
    uint64_t *v_full = bars + 2 * kStages, *v_empty = bars + 3 * kStages;
    uint64_t *q_full = bars + 4 * kStages, *q_empty = q_full + 1;
    uint64_t *s_full = q_empty + 1, *s_empty = s_full + kSBufs, *p_full = s_empty + kSBufs;
    uint64_t *o_empty = p_full + kSBufs, *o_final = o_empty + 1;
    uint64_t *xm_bar = o_final + 1;          // [2 slots][4 row quarters], pair max exchange
    uint64_t *xl_bar = xm_bar + 8;           // [4 row quarters], pair row-sum exchange
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Ly::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Ly::kMisc + 4);

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort_flag) post_status(A.status, KV_ERR_UNSUPPORTED);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int b = 0; b < kSBufs; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 1);
            mbar_init(&p_full[b], kSoftWarps);
        }
        mbar_init(o_empty, kSoftWarps);
        mbar_init(o_final, 1);
        for (int b = 0; b < 8; ++b) mbar_init(&xm_bar[b], 2);
        for (int b = 0; b < 4; ++b) mbar_init(&xl_bar[b], 2);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
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
            // L2 prefetch cursor: walks the same (item, tile) sequence as the loads,
            // kPrefetchTiles tiles ahead of them, so the smem ring's loads hit L2.
            long long pf_item = blockIdx.x, pf_row0 = 0;
            int pf_t = 0, pf_end = 0;
            auto pf_open = [&]() {
                if (pf_item < A.total_items) {
                    const Item pi = decode_item(pf_item, A, P);
                    pf_row0 = unit_info(P, pi.u, P.cu).kv_row0;
                    pf_t = pi.t0;
                    pf_end = pi.t1;
                }
            };
            auto pf_step = [&]() {
                if (pf_item >= A.total_items) return;
                const int ky = (int)(pf_row0 + (long long)pf_t * kTileKeys);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_prefetch_2d(&tm_k, kb * 64, ky);
                    tma_prefetch_2d(&tm_v, kb * 64, ky);
                }
                if (++pf_t >= pf_end) {
                    pf_item += gridDim.x;
                    pf_open();
                }
            };
            pf_open();
            for (int i = 0; i < kPrefetchTiles; ++i) pf_step();
            for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
                const Item it = decode_item(item, A, P);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                ok = mbar_wait(q_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, kWaitNs);
                if (!ok) break;
                mbar_arrive_expect_tx(q_full, Ly::kOp);
                const int qy = (int)(U.q_row0 + it.c * kChunkRows);
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb)
                    tma_load_2d(smem + Ly::kQ + kb * kBlockBytes, &tm_q, q_full, kb * 64, qy);
                for (int t = it.t0; ok && t < it.t1; ++t, ++tcount) {
                    const int s = (int)(tcount % kStages);
                    const uint32_t par = (uint32_t)((tcount / kStages) & 1) ^ 1u;
                    const int ky = (int)(U.kv_row0 + (long long)t * kTileKeys);
                    pf_step();
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
            const uint32_t idesc_s = idesc_bf16_f32(128, kTileKeys);
            const uint32_t idesc_pv = idesc_bf16_f32_bmn(128, D);
            const uint64_t qa0 = sdesc_k_sw128(smem_u32(smem + Ly::kQ));
            long long tcount = 0, icount = 0;
            bool ok = true;
            // O += P_hi V + P_lo V for global tile tc (the item's first tile overwrites O)
            auto pv = [&](long long tc, bool first) {
                const int s = (int)(tc % kStages);
                const int b = (int)(tc % kSBufs);
                if (first)
                    ok = ok && mbar_wait(o_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, kWaitNs);
                ok = ok && mbar_wait(&p_full[b], (uint32_t)((tc / kSBufs) & 1), abort_flag, kWaitNs);
                ok = ok && mbar_wait(&v_full[s], (uint32_t)((tc / kStages) & 1), abort_flag,
                                     kWaitNs);
                if (!ok) return;
                tc_fence_after();
                const uint64_t vb =
                    sdesc_mn_sw128(smem_u32(smem + Ly::kV + s * Ly::kOp), kBlockBytes);
                const uint32_t pcol = tmem + b * kTileKeys;
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int q = 0; q < kTileKeys / 16; ++q) {
                        // keys 16q..16q+15: P_hi in columns 16q..16q+7, P_lo in 16q+8..16q+15
                        const uint32_t a = pcol + q * 16 + part * 8;
                        const uint64_t bd = sdesc_add(vb, q * 16 * 128);
                        if (part == 0 && q == 0 && first)
                            mma_ts_c<false>(tmem + kOCol, a, bd, idesc_pv);
                        else
                            mma_ts_c<true>(tmem + kOCol, a, bd, idesc_pv);
                    }
                mma_commit(&s_empty[b]);
                mma_commit(&v_empty[s]);
            };
            for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
                const Item it = decode_item(item, A, P);
                const int ntiles = it.t1 - it.t0;
                ok = mbar_wait(q_full, (uint32_t)(icount & 1), abort_flag, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                for (int i = 0; ok && i < ntiles; ++i) {
                    const long long tc = tcount + i;
                    const int b = (int)(tc % kSBufs);
                    const int s = (int)(tc % kStages);
                    ok = mbar_wait(&s_empty[b], (uint32_t)((tc / kSBufs) & 1) ^ 1u, abort_flag,
                                   kWaitNs) &&
                         mbar_wait(&k_full[s], (uint32_t)((tc / kStages) & 1), abort_flag, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kb0 = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
                    const uint32_t d_s = tmem + b * kTileKeys;
                    mma_ss_c<false>(d_s, qa0, kb0, idesc_s);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            if (kb | kk)
                                mma_ss_c<true>(d_s, sdesc_add(qa0, ko), sdesc_add(kb0, ko), idesc_s);
                        }
                    mma_commit(&s_full[b]);
                    mma_commit(&k_empty[s]);
                    if (i > 0) pv(tc - 1, i == 1);
                }
                if (ok && ntiles > 0) pv(tcount + ntiles - 1, ntiles == 1);
                mma_commit(o_final);
                mma_commit(q_empty);
                tcount += ntiles;
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
        }
    } else if (run) {
        // ------------------------------------------------------------ softmax
        const int ew = warp - 2;
        const int half = ew >> 2;
        const int quarter = warp & 3;
        const int rr = quarter * 32 + lane;               // row of the chunk = TMEM lane
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float *xmax = reinterpret_cast<float *>(smem + Ly::kXmax);
        float *xl = reinterpret_cast<float *>(smem + Ly::kXl);
        const float cs = P.scale_log2;
        constexpr int kHalfKeys = kTileKeys / 2;
        constexpr int kHalfD = D / 2;
        long long tcount = 0, icount = 0;
        bool ok = true;
        for (long long item = blockIdx.x; ok && item < A.total_items; item += gridDim.x) {
            const Item it = decode_item(item, A, P);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int ntiles = it.t1 - it.t0;
            const int row = it.c * kChunkRows + rr;
            const bool row_valid = row < P.rows;
            const int pos = U.n - P.w + (row % P.w);
            const int pos_min = U.n - P.w;
            float m_used = -INFINITY, l = 0.f;
            for (int i = 0; ok && i < ntiles; ++i) {
                const long long tc = tcount + i;
                const int b = (int)(tc % kSBufs);
                const int kt = (it.t0 + i) * kTileKeys;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (uint32_t)((tc / kSBufs) & 1),
                                                       abort_flag, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                const int j0 = half * kHalfKeys;
                const uint32_t s_col = tmem + lane_addr + b * kTileKeys + j0;
                // causal mask (only the tiles that reach into the window need it)
                const bool boundary = kt + kTileKeys - 1 > pos_min;
                const int lim = row_valid ? (boundary ? pos - kt : kTileKeys - 1) : -1;
                // warp-uniform: the mask code only runs on tiles that need it
                const bool masked = __any_sync(0xffffffffu, lim < kTileKeys - 1);
                // row max over this warp's 64 keys, 16 columns at a time
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                for (int c = 0; c < kHalfKeys / 16; ++c) {
                    float sv[16];
                    tmem_ld16(s_col + c * 16, sv);
                    tmem_ld_wait();
                    reg_fence(sv);
                    if (masked) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float x = (j0 + c * 16 + j > lim) ? -INFINITY : sv[j];
                            mx4[j & 3] = fmaxf(mx4[j & 3], x);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], sv[j]);
                    }
                }
                const float mh = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                float *slot = xmax + (int)(tc & 1) * 256;
                slot[half * 128 + rr] = mh;
                __syncwarp();
                uint64_t *xb = &xm_bar[(int)(tc & 1) * 4 + quarter];
                if (lane == 0) mbar_arrive(xb);
                ok = __all_sync(0xffffffffu, mbar_wait(xb, (uint32_t)((tc >> 1) & 1), abort_flag,
                                                       kWaitNs));
                if (!ok) break;
                const float mx = fmaxf(mh, slot[(half ^ 1) * 128 + rr]);
                const float m_tile = mx * cs;
                const bool need = m_tile > m_used + kRescaleLog2;
                const float factor = need ? ex2_approx(m_used - m_tile) : 1.f;
                if (__any_sync(0xffffffffu, need && i > 0)) {
                    // O holds P V of earlier tiles: rescale it once P V of tile tc-1 is done.
                    // That P V frees tile tc-1's S/P buffer; the previous phase of that
                    // barrier (P V of tc-1-kSBufs) is known done, so this cannot alias.
                    const long long tp = tc - 1;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&s_empty[(int)(tp % kSBufs)],
                                              (uint32_t)((tp / kSBufs) & 1), abort_flag, kWaitNs));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kHalfD / 16; ++c) {
                        float o[16];
                        const uint32_t oc = tmem + lane_addr + kOCol + half * kHalfD + c * 16;
                        tmem_ld16(oc, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] *= factor;
                        tmem_st16(oc, o);
                    }
                }
                if (need) {
                    l *= factor;
                    m_used = m_tile;
                }
                // P over the S columns just read: each 16-key chunk's own 16 columns
                // take its P_hi (first 8) and P_lo (last 8)
                float2 lsum = make_float2(0.f, 0.f);
                const float negm = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll 1
                for (int c = 0; c < kHalfKeys / 16; ++c) {
                    float sv[16];
                    const uint32_t col = s_col + c * 16;
                    tmem_ld16(col, sv);
                    tmem_ld_wait();
                    reg_fence(sv);
                    if (masked)
                        soft16_tmem<true>(sv, j0 + c * 16, lim, cs, negm, lsum, col, col + 8);
                    else
                        soft16_tmem<false>(sv, j0 + c * 16, lim, cs, negm, lsum, col, col + 8);
                }
                l += lsum.x + lsum.y;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;
            // item end: read O once the last P V is done, write this split's partial
            const size_t prow_idx = (((size_t)it.u * P.max_splits + it.split) * P.rows) + row;
            if (ntiles > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(o_final, (uint32_t)(icount & 1), abort_flag, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                float *po = A.part_o + prow_idx * D + half * kHalfD;
#pragma unroll
                for (int c = 0; c < kHalfD / 16; ++c) {
                    float o[16];
                    tmem_ld16(tmem + lane_addr + kOCol + half * kHalfD + c * 16, o);
                    tmem_ld_wait();
                    reg_fence(o);
                    if (row_valid) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(po + c * 16 + j) =
                                make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
            }
            // the row sum is split between the pair: half 1 hands its part to half 0
            if (half == 1) xl[rr] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&xl_bar[quarter]);
            ok = __all_sync(0xffffffffu, mbar_wait(&xl_bar[quarter], (uint32_t)(icount & 1),
                                                   abort_flag, kWaitNs));
            if (!ok) break;
            if (half == 0 && row_valid) A.part_ml[prow_idx] = make_float2(m_used, l + xl[rr]);
            tcount += ntiles;
            ++icount;
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

template <int D>
cudaError_t attention_d(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                        const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const long long q_rows = (long long)P.R * P.L * P.Hq * P.w;
    const long long kv_rows = (long long)P.L * P.H * P.N_tot;
    if (!make_tile_map(&mq, q, q_rows, D) || !make_tile_map(&mk, k, kv_rows, D) ||
        !make_tile_map(&mv, v, kv_rows, D))
        return cudaErrorInvalidValue;
    launch_plan(P, kSplitKeys, ws.plan, st);
    AttnArgs A;
    A.plan = ws.plan;
    A.part_ml = ws.part_ml;
    A.part_o = ws.part_o;
    A.chunks = ws.chunks;
    A.total_items = total_blocks(P, kSplitKeys) * ws.chunks;
    A.status = ws.status;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = Layout<D>::kTotal;
    cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const long long grid = std::min<long long>(sms, A.total_items);
    if (grid > 0) attn_tc_kernel<D><<<(unsigned)grid, kThreads, smem, st>>>(P, mq, mk, mv, A);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_partials(const DevProblem &P, const __nv_bfloat16 *q,
                                      const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                      const ScoreWs &ws, cudaStream_t s) {
    return P.d == 64 ? attention_d<64>(P, q, k, v, ws, s) : attention_d<128>(P, q, k, v, ws, s);
}

}  // namespace kvevict
