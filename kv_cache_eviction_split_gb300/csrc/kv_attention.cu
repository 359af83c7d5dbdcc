// kv_attention.cu -- pass 1 of the DropKV score on the tcgen05 tensor cores:
// causal window attention over each unit's keys, split across CTAs (split-K),
// producing per split the row max m (log2 units), the row sum l of
// 2^(s*scale*log2 e - m) and the unnormalised output O = sum_j P_j v_j.  The
// merge in kv_score.cu combines the splits (DropKV, "Methodology in Plain
// English": the attention output a whose removal shift the score measures).
//
// Query-major, one 128-row chunk of the unit's G*w window rows per work item:
//   S = Q K^T    M = 128 rows, N = 128 keys, K = d     (fp32 in TMEM, 2 buffers)
//   O += P V     M = 128 rows, N = d, K = 128 keys     (fp32 in TMEM; V is the
//                MN-major B operand; the softmax warps write P to swizzled
//                shared memory as two bf16 halves P_hi = bf16(p) and
//                P_lo = bf16(p - P_hi), and O accumulates P_hi V + P_lo V)
// A single bf16 P leaves a with ~2^-9 relative error, which the rescoring
// expansion amplifies where a is close to a value row (short requests,
// concentrated attention); the split keeps ~16 bits of p.
// The softmax warps own one row each: tile max with the causal mask, a lazy
// rescale (O and l are rescaled only when the tile max exceeds the running
// max by more than 2^8, so the running max may trail the true max by at most
// 8 in log2 units -- every exponent stays <= 2^8), p = 2^(s*c - m), row sums
// from the unrounded fp32 p.
//
// Barrier parities are tracked from use counts; no barrier can run more than
// one phase ahead of its waiter.  The P buffer is single: the softmax warps
// write P of tile i only after P V of tile i-1 is done, which is also the
// moment O may be rescaled.
//
// Warp roles (320 threads): warp 0 TMA producer (Q chunk per item, K and V
// tiles through a 2-stage ring); warp 1 TMEM owner and MMA issuer, running
// S of tile i+1 ahead of P V of tile i; warps 2-9 softmax, two per row.  Work items are
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
constexpr int kStages = 2;
constexpr int kSoftWarps = 8;    // two per row quarter, each on half of a tile's keys
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kBlockBytes = 128 * 128;       // [128 rows][64 bf16], 128 B swizzle
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct Layout {
    static constexpr int kOp = (D / 64) * kBlockBytes;   // [128][D] bf16
    static constexpr int kPbuf = 2 * kBlockBytes;        // [128 rows][128 keys] bf16 (hi, then lo)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kOp;
    static constexpr int kV = kK + kStages * kOp;
    static constexpr int kP = kV + kStages * kOp;
    static constexpr int kXmax = kP + 2 * kPbuf;          // [2 slots][2 halves][128] float
    static constexpr int kXl = kXmax + 2 * 2 * 128 * 4;    // [128] float
    static constexpr int kBars = kXl + 128 * 4;
    static constexpr int kNumBars = 4 * kStages + 2 + 4 + 2 + 2 + 8 + 4;
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

// Running maxima (4 independent chains) of 16 logits; keys past `lim` excluded.
__device__ __forceinline__ void tile_max16(const float (&v)[16], int j0, int lim, bool masked,
                                           float (&mx)[4]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float x = (masked && j0 + j > lim) ? -INFINITY : v[j];
        mx[j & 3] = fmaxf(mx[j & 3], x);
    }
}

// p = 2^(s c - m) for 16 keys (two 8-key groups of the P tile): adds p to the
// row sum and stores bf16(p) to the P_hi tile and bf16(p - P_hi) to the P_lo
// tile (kPbuf bytes later), in the 128-byte swizzled K-major layout.
template <int kPbuf>
__device__ __forceinline__ void soft16(const float (&v)[16], int j0, int lim, bool masked,
                                       float cs, float negm, float2 &lsum, uint8_t *prow, int rr) {
    const float2 cs2 = make_float2(cs, cs);
    const float2 nm2 = make_float2(negm, negm);
    const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int g8 = 0; g8 < 2; ++g8) {
        uint32_t whi[4], wlo[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int j = g8 * 8 + 2 * h;
            const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), cs2, nm2);
            float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            if (masked) {
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
        const int ch = (j0 >> 3) + g8;    // 8-key chunk of the 128-key row
        const int off = (ch >> 3) * kBlockBytes + (((ch & 7) ^ (rr & 7)) << 4);
        *reinterpret_cast<uint4 *>(prow + off) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
        *reinterpret_cast<uint4 *>(prow + kPbuf + off) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
    }
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
    uint64_t *s_full = q_empty + 1, *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2, *p_empty = p_full + 1;
    uint64_t *o_empty = p_empty + 1, *o_final = o_empty + 1;
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
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], kSoftWarps);
        }
        mbar_init(p_full, kSoftWarps);
        mbar_init(p_empty, 1);
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
            const uint32_t q_base = smem_u32(smem + Ly::kQ);
            long long tcount = 0, icount = 0;
            bool ok = true;
            // O += P_hi V + P_lo V for global tile tc (the item's first tile overwrites O)
            auto pv = [&](long long tc, bool first) {
                const int s = (int)(tc % kStages);
                if (first)
                    ok = ok && mbar_wait(o_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, kWaitNs);
                ok = ok && mbar_wait(p_full, (uint32_t)(tc & 1), abort_flag, kWaitNs);
                ok = ok && mbar_wait(&v_full[s], (uint32_t)((tc / kStages) & 1), abort_flag,
                                     kWaitNs);
                if (!ok) return;
                tc_fence_after();
                const uint64_t vb = sdesc_mn_sw128(smem_u32(smem + Ly::kV + s * Ly::kOp), kBlockBytes);
                const uint64_t pa0 = sdesc_k_sw128(smem_u32(smem + Ly::kP));
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_add(pa0, part * Ly::kPbuf + kb * kBlockBytes + kk * 32);
                            const uint64_t b = sdesc_add(vb, (kb * 64 + kk * 16) * 128);
                            if (part == 0 && kb == 0 && kk == 0 && first)
                                mma_ss_c<false>(tmem + kOCol, a, b, idesc_pv);
                            else
                                mma_ss_c<true>(tmem + kOCol, a, b, idesc_pv);
                        }
                mma_commit(p_empty);
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
                    const int sb = (int)(tc & 1);
                    const int s = (int)(tc % kStages);
                    ok = mbar_wait(&s_empty[sb], (uint32_t)((tc >> 1) & 1) ^ 1u, abort_flag,
                                   kWaitNs) &&
                         mbar_wait(&k_full[s], (uint32_t)((tc / kStages) & 1), abort_flag, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kb0 = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
                    const uint64_t qa0 = sdesc_k_sw128(q_base);
                    const uint32_t d_s = tmem + sb * kTileKeys;
                    mma_ss_c<false>(d_s, qa0, kb0, idesc_s);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            if (kb | kk)
                                mma_ss_c<true>(d_s, sdesc_add(qa0, ko), sdesc_add(kb0, ko), idesc_s);
                        }
                    mma_commit(&s_full[sb]);
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
        // Warps w and w+4 own the same 32 rows (TMEM lane quarter w % 4); warp
        // half 0 takes keys 0-63 of every tile, half 1 keys 64-127, and O columns
        // split the same way.  They agree on the row max through shared memory.
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
                const int sb = (int)(tc & 1);
                const int kt = (it.t0 + i) * kTileKeys;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (uint32_t)((tc >> 1) & 1),
                                                       abort_flag, kWaitNs));
                if (!ok) break;
                tc_fence_after();
                const int j0 = half * kHalfKeys;
                const uint32_t s_col = tmem + lane_addr + sb * kTileKeys + j0;
                // causal mask (only the tiles that reach into the window need it)
                const bool boundary = kt + kTileKeys - 1 > pos_min;
                const int lim = row_valid ? (boundary ? pos - kt : kTileKeys - 1) : -1;
                const bool masked = lim < kTileKeys - 1;
                // pass A: row max over this warp's 64 keys, then over the pair
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                {
                    float bA[16], bB[16];
                    tmem_ld16(s_col, bA);
#pragma unroll
                    for (int c = 0; c < kHalfKeys / 16; c += 2) {
                        tmem_ld_wait();
                        reg_fence(bA);
                        tmem_ld16(s_col + (c + 1) * 16, bB);
                        tile_max16(bA, j0 + c * 16, lim, masked, mx4);
                        tmem_ld_wait();
                        reg_fence(bB);
                        if (c + 2 < kHalfKeys / 16) tmem_ld16(s_col + (c + 2) * 16, bA);
                        tile_max16(bB, j0 + (c + 1) * 16, lim, masked, mx4);
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
                // the P buffer is free once P V of tile tc-1 is done; O is then stable
                ok = __all_sync(0xffffffffu, mbar_wait(p_empty, (uint32_t)(tc & 1) ^ 1u,
                                                       abort_flag, kWaitNs));
                if (!ok) break;
                if (__any_sync(0xffffffffu, need && i > 0)) {
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
                    tmem_st_wait();
                }
                if (need) {
                    l *= factor;
                    m_used = m_tile;
                }
                // pass B: p = 2^(s c - m), row sum, P_hi / P_lo to shared memory
                uint8_t *prow = smem + Ly::kP + rr * 128;
                float2 lsum = make_float2(0.f, 0.f);
                const float negm = m_used == -INFINITY ? 0.f : -m_used;
                {
                    float bA[16], bB[16];
                    tmem_ld16(s_col, bA);
#pragma unroll
                    for (int c = 0; c < kHalfKeys / 16; c += 2) {
                        tmem_ld_wait();
                        reg_fence(bA);
                        tmem_ld16(s_col + (c + 1) * 16, bB);
                        soft16<Ly::kPbuf>(bA, j0 + c * 16, lim, masked, cs, negm, lsum, prow, rr);
                        tmem_ld_wait();
                        reg_fence(bB);
                        if (c + 2 < kHalfKeys / 16) tmem_ld16(s_col + (c + 2) * 16, bA);
                        soft16<Ly::kPbuf>(bB, j0 + (c + 1) * 16, lim, masked, cs, negm, lsum, prow,
                                          rr);
                    }
                }
                l += lsum.x + lsum.y;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
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
