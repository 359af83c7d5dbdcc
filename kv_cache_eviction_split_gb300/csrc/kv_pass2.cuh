// kv_pass2.cuh -- pass 2 of the DropKV score on the tcgen05 tensor cores.
//
// For every key j of a unit and every window row r that sees it (score rule
// KV_SCORE_DROPKV):
//     s   = q_r . k_j                         (tensor core, fp32 in TMEM)
//     X   = (a_hi_r + a_lo_r) . v_j           (tensor core, two bf16 MMAs)
//     p   = 2^(s * scale * log2 e - m_r - log2 l_r)     (= e / l_r)
//     x   = ||a_r||^2 - 2 X + ||v_j||^2      = ||a_r - v_j||^2 (the expansion the
//                                              DropKV scoring-kernel description uses)
//     S_j += p / (1 - p) * sqrt(x)           = p/(1-p) * ||a_r - v_j||
// (DropKV, Key Contributions 1 and Methodology in Plain English).  a = a_hi +
// a_lo is the pass-1 output split into two bf16 halves, so the expansion keeps
// ~16 bits of a instead of bf16's 8.
//
// The other rules change only the term: KV_SCORE_DROPKV_SQUARED adds the
// square of the same term, (p/(1-p))^2 x (DropKV, "Methodology in Plain
// English": the window sum taken squared), and KV_SCORE_ATTN_SUM adds p alone
// (PyramidKV guide, "Observation Window and Aggregated Attention Eviction").
// The attention sum needs neither V nor a: its kernel loads only Q and K,
// issues only S = K Q^T, and runs four K stages and four TMEM buffers.
//
// Orientation is key-major: one MMA tile is 128 keys (M, TMEM lanes) by the
// rows of a 128-row chunk of the unit's window rows (N).  The epilogue reads
// TMEM in the 16x256b shape, so each thread holds two keys and a fixed set of
// 32 rows: the per-row statistics stay in registers for the whole work item
// and the inner loop touches no shared memory (the SS MMAs keep the shared
// memory data path busy, and loads issued behind them wait long).  Work items
// = (unit, 64-key-tile block, row chunk); a persistent grid walks them
// round-robin, chunk fastest, so the chunks of one key block run on
// neighbouring SMs at the same time and share K/V through L2.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: the chunk's Q, a_hi, a_lo once per item; K and V
//               tiles through a 2-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread): per tile S = K Q^T and
//               X = V a_hi^T + V a_lo^T over all rows of the chunk, into one of
//               two TMEM buffers, so tile i+1 computes while tile i is scored
//               and a K/V stage frees as soon as its MMAs complete (||v_j||^2
//               comes from pass 1, which computes it while converting V)
//   warps 2-9   epilogue: warp w reads TMEM lanes 32 (w % 4) + 16 h .. +15
//               (h = 0 for warps 2-5, 1 for 6-9) over all rows of the chunk;
//               the four threads that share a key add their sums by shuffles
// Every wait is bounded: on expiry the kernel posts KV_ERR_TIMEOUT, the other
// roles drain out, TMEM is freed and the kernel returns.
//
// The pass is written as a device body (rescore_body) that the stand-alone
// kernel in kv_rescore.cu and the fused kernel in kv_fused.cu call with their
// CTA index and count.
#pragma once
#include <cfloat>

#include "kv_internal.cuh"
#include "kv_sm100.cuh"

namespace kvevict {
namespace pass2 {
using namespace sm100;

constexpr int kTileKeys = 128;
constexpr int kChunkRows = 128;
constexpr int kTilesPerItem = 64;
constexpr int kPrefetchTiles = 2;   // K/V tiles requested into L2 ahead of the smem loads
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kBlockBytes = kChunkRows * 128;   // one [128 rows][64 bf16] swizzled box
static_assert(kTileKeys * kTilesPerItem == kPass2BlockKeys, "pass-2 item order tables");

template <int D, int RULE>
struct Layout {
    static constexpr bool kX = RULE != KV_SCORE_ATTN_SUM;  // X = a . v (and V) needed
    static constexpr int kOp = (D / 64) * kBlockBytes;     // one [128][D] bf16 operand
    static constexpr int kKSt = kX ? 2 : 4;                // K stages
    static constexpr int kVSt = kX ? 2 : 0;                // V stages
    static constexpr int kQ = 0;
    static constexpr int kAhi = kQ + kOp;
    static constexpr int kAlo = kAhi + (kX ? kOp : 0);
    static constexpr int kK = kAlo + (kX ? kOp : 0);
    static constexpr int kV = kK + kKSt * kOp;
    static constexpr int kBars = kV + kVSt * kOp;
    static constexpr int kBufs = kX ? 2 : 4;               // TMEM buffers (S, X) or S
    static constexpr int kBufCols = kX ? 256 : 128;
    static constexpr int kNumBars = 2 * kKSt + 2 * (kVSt > 0 ? kVSt : 1) + 2 + 2 * kBufs + 1;
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kTotal = kMisc + 16;
};

struct RescoreArgs {
    const int32_t *plan;       // [units + 1] prefix of key-tile blocks per unit
    const float2 *stat_ml;     // [units][rows] (m in log2 units, l)
    const float *stat_a2;      // [units][rows]
    const float *v2;           // [L*H*N_tot] ||v_j||^2 (from pass 1)
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

// Work item `item` of a grid of `ncta` CTAs.  Chunks run fastest, so the chunks
// of one key block sit in one round of the grid.  When ncta is a multiple of the
// chunk count, a CTA meets the same chunk in every round; with a short last chunk
// (448 rows = 3 x 128 + 64) the CTAs that always get it idle at the end, so the
// chunk is then rotated by the round, which keeps the mapping one-to-one (the
// rotation is the same for all chunks of a block) and gives every CTA every chunk
// in turn (448 rows: pass 2 4.61 -> 4.53 ms; with equal chunks it is not applied).
__device__ __forceinline__ Item decode_item(long long item, long long ncta, const RescoreArgs &A,
                                            const DevProblem &P, const ItemOrder &O) {
    Item it;
    it.c = (int)(item % A.chunks);
    if (P.rows % kChunkRows != 0 && ncta % A.chunks == 0)
        it.c = (int)((it.c + item / ncta) % A.chunks);
    const long long gb = item / A.chunks;
    long long lo = 0;
    int blk = 0;
    if (O.nrun > 0) {           // full blocks first, then partial ones
        order_decode(O, gb, lo, blk);
    } else {                    // many runs of lengths: plan[lo] <= gb < plan[lo + 1]
        long long hi = P.units;
        while (hi - lo > 1) {
            const long long mid = (lo + hi) >> 1;
            if (A.plan[mid] <= gb) lo = mid; else hi = mid;
        }
        blk = (int)(gb - A.plan[lo]);
    }
    it.u = lo;
    const int n = (int)(P.cu[(int)(lo / ((long long)P.L * P.H)) + 1] -
                        P.cu[(int)(lo / ((long long)P.L * P.H))]);
    const int tiles = (n + kTileKeys - 1) / kTileKeys;
    it.t_begin = blk * kTilesPerItem;
    it.t_end = min(it.t_begin + kTilesPerItem, tiles);
    return it;
}

// Rows of chunk c rounded up to a multiple of 32 (the MMA N and the TMEM columns used).
__device__ __forceinline__ int chunk_rows_n(const DevProblem &P, int c) {
    const int rc = min(kChunkRows, P.rows - c * kChunkRows);
    return ((rc + 31) / 32) * 32;
}

// ||v_j||^2: read-only (non-coherent) load, or a plain one when the value was
// written earlier in the same kernel.
template <bool kCoherent>
__device__ __forceinline__ float ld_v2(const float *p) {
    if constexpr (kCoherent) return *p;
    else return __ldg(p);
}

// One (row pair, key) term pair.  p = 2^(s c - m'); `vis` = 0 drops a row that
// does not see the key.  KV_SCORE_DROPKV adds p/(1 - p) * sqrt(x) with
// x = |||a||^2 - 2X + ||v||^2|, written as p * x * rsqrt((1 - p)^2 x + tiny)
// so one MUFU op gives sqrt(x)/(1-p) and x = 0 gives 0; the squared rule adds
// the square of that term; the attention sum adds p.  The expansion can round
// below zero only where ||a - v||^2 is within its rounding error of zero; the
// absolute value keeps the term real and non-negative there, as a clamp at zero
// would, with no min/max instructions (the epilogue is bound by its instruction
// issue: 5.90 -> 5.50 ms for this pass at 256 window rows).
template <int RULE>
__device__ __forceinline__ void term_pair(float2 sp, float2 xp, float2 nm, float2 a2, float2 v2,
                                          float cscale, float2 &acc, bool vis0 = true,
                                          bool vis1 = true) {
    const float2 t = __ffma2_rn(sp, make_float2(cscale, cscale), nm);
    float2 pr = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    if (!vis0) pr.x = 0.f;
    if (!vis1) pr.y = 0.f;
    if constexpr (RULE == KV_SCORE_ATTN_SUM) {
        acc = __fadd2_rn(acc, pr);
    } else {
        const float2 den = __ffma2_rn(pr, make_float2(-1.f, -1.f), make_float2(1.f, 1.f));
        const float2 av = __fadd2_rn(a2, v2);
        float2 x = __ffma2_rn(xp, make_float2(-2.f, -2.f), av);
        x.x = fabsf(x.x);
        x.y = fabsf(x.y);
        const float2 y = __ffma2_rn(__fmul2_rn(den, den), x, make_float2(1e-30f, 1e-30f));
        const float2 px = __fmul2_rn(pr, x);
        const float2 rs = make_float2(rsqrt_approx(y.x), rsqrt_approx(y.y));
        if constexpr (RULE == KV_SCORE_DROPKV_SQUARED) {
            const float2 tr = __fmul2_rn(px, rs);
            acc = __ffma2_rn(tr, tr, acc);
        } else {
            acc = __ffma2_rn(px, rs, acc);
        }
    }
}

// Adds the terms of one 32-column group for the thread's two keys: sv / xv are
// 16x256b.x4 loads of S and X (v[4r], v[4r+1]: key 0, rows 2 part + 8r + {0,1};
// v[4r+2], v[4r+3]: key 1, the same rows).  Every row sees both keys.
template <int RULE>
__device__ __forceinline__ void rescore_x4(const float (&sv)[16], const float (&xv)[16],
                                           const float2 *nm, const float2 *a2, float cscale,
                                           const float2 (&v2)[2], float2 (&acc)[2]) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int k = 0; k < 2; ++k)
            term_pair<RULE>(make_float2(sv[4 * r + 2 * k], sv[4 * r + 2 * k + 1]),
                            make_float2(xv[4 * r + 2 * k], xv[4 * r + 2 * k + 1]), nm[r], a2[r],
                            v2[k], cscale, acc[k]);
}

// -m' = -(m + log2 l) and ||a||^2 of one unit-local row; padding rows (>= rows)
// get p = 0.
__device__ __forceinline__ void row_stats(const float2 *ml, const float *a2, int row, int rows,
                                          float &nm, float &aa) {
    if (row < rows) {
        const float2 v = ml[row];
        nm = -(v.x + log2f(v.y));
        aa = a2[row];
    } else {
        nm = -INFINITY;
        aa = 0.f;
    }
}

// As rescore_x4 for a tile that reaches the observation window, where a row at
// window slot t sees key j only when j - (n - w) <= t (jrel[k] = j_k - (n - w)).
// Recomputes the row statistics from the unit's arrays (row0 = unit-local row of
// pair 0): this path runs for one or two tiles per unit, in a loop of its own so
// the masks stay out of the unrolled code of the other tiles.
template <int RULE>
__device__ __forceinline__ void rescore_x4_window(const float (&sv)[16], const float (&xv)[16],
                                               const float2 *ml, const float *a2g, int rows,
                                               int row0, int w, const int (&jrel)[2],
                                               float cscale, const float2 (&v2)[2],
                                               float2 (&acc)[2]) {
    for (int r = 0; r < 4; ++r) {
        const int row = row0 + 8 * r;
        float n0, n1, q0, q1;
        row_stats(ml, a2g, row, rows, n0, q0);
        row_stats(ml, a2g, row + 1, rows, n1, q1);
        const int rm0 = row % w;
        const int rm1 = rm0 + 1 == w ? 0 : rm0 + 1;
        for (int k = 0; k < 2; ++k)
            term_pair<RULE>(make_float2(sv[4 * r + 2 * k], sv[4 * r + 2 * k + 1]),
                            make_float2(xv[4 * r + 2 * k], xv[4 * r + 2 * k + 1]),
                            make_float2(n0, n1), make_float2(q0, q1), v2[k], cscale, acc[k],
                            jrel[k] <= rm0, jrel[k] <= rm1);
    }
}

// The kernel body, for CTA `cta` of `ncta` (all threads of the CTA call it;
// `tmem` is the base of 512 TMEM columns the caller allocated; warps from
// 2 + kEpiWarps on idle).  kCoherent reads ||v||^2 with coherent loads, for
// callers that wrote it earlier in the same kernel.
template <int D, int RULE, bool kCoherent = false>
__device__ __forceinline__ void rescore_body(const DevProblem P, const CUtensorMap *tm_q,
                                             const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                             const CUtensorMap *tm_ahi, const CUtensorMap *tm_alo,
                                             const RescoreArgs A, const ItemOrder &ord,
                                             uint8_t *smem, uint32_t tmem, long long cta,
                                             long long ncta) {
    using Ly = Layout<D, RULE>;
    constexpr bool kX = Ly::kX;
    constexpr int kKSt = Ly::kKSt;
    constexpr int kVSt = kX ? Ly::kVSt : 1;   // barrier slots (unused without X)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly::kBars);
    uint64_t *k_full = bars, *k_empty = bars + kKSt;
    uint64_t *v_full = bars + 2 * kKSt, *v_empty = v_full + kVSt;
    uint64_t *qa_full = v_empty + kVSt, *qa_empty = qa_full + 1;
    constexpr int kBufs = Ly::kBufs;
    uint64_t *tm_full = qa_empty + 1, *tm_empty = tm_full + kBufs;
    uint64_t *mma_done = tm_empty + kBufs;   // the MMA thread's last MMAs are done (exit)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Ly::kMisc + 4);

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort_flag) post_status(A.status, KV_ERR_UNSUPPORTED);
        for (int s = 0; s < kKSt; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVSt; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(qa_full, 1);
        mbar_init(qa_empty, 1);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&tm_full[h], 1);
            mbar_init(&tm_empty[h], kEpiWarps);
        }
        for (int h = 2; h < kBufs; ++h) {
            mbar_init(&tm_full[h], 1);
            mbar_init(&tm_empty[h], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(tm_q);
        prefetch_tensormap(tm_k);
        prefetch_tensormap(tm_v);
        prefetch_tensormap(tm_ahi);
        prefetch_tensormap(tm_alo);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool run = *abort_flag == 0;

    if (run && warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            long long tcount = 0, icount = 0;
            long long qcount = 0, kiss = 0, viss = 0;   // Q/a, K and V loads issued
            bool ok = true;
            // L2 prefetch cursor: walks the same (item, tile) sequence as the loads,
            // kPrefetchTiles tiles ahead of them, so the smem ring's loads hit L2.
            long long pf_item = cta, pf_row0 = 0;
            int pf_t = 0, pf_end = 0;
            auto pf_open = [&]() {
                if (pf_item < A.total_items) {
                    const Item pi = decode_item(pf_item, ncta, A, P, ord);
                    pf_row0 = unit_info(P, pi.u, P.cu).kv_row0;
                    pf_t = pi.t_begin;
                    pf_end = pi.t_end;
                }
            };
            auto pf_step = [&]() {
                if (pf_item >= A.total_items) return;
                const int ky = (int)(pf_row0 + (long long)pf_t * kTileKeys);
                if (!in_range(ky, kv_rows_total(P), A.status)) {
                    pf_item = A.total_items;   // no further prefetches
                    return;
                }
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_prefetch_2d(tm_k, kb * 64, ky);
                    if constexpr (kX) tma_prefetch_2d(tm_v, kb * 64, ky);
                }
                if (++pf_t >= pf_end) {
                    pf_item += ncta;
                    pf_open();
                }
            };
            pf_open();
            for (int i = 0; i < kPrefetchTiles; ++i) pf_step();
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, ncta, A, P, ord);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                ok = mbar_wait(qa_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, P.wait_ns);
                if (!ok) break;
                mbar_arrive_expect_tx(qa_full, (kX ? 3 : 1) * Ly::kOp);
                const int qy = (int)(U.q_row0 + it.c * kChunkRows);
                const int ay = (int)(it.u * A.a_rows + it.c * kChunkRows);
                if (!in_range(qy, q_rows_total(P), A.status) ||
                    !in_range(ay, P.units * A.a_rows, A.status))
                    ok = false;
#pragma unroll
                for (int kb = 0; kb < D / 64; ++kb) {
                    tma_load_2d(smem + Ly::kQ + kb * kBlockBytes, tm_q, qa_full, kb * 64, qy);
                    if constexpr (kX) {
                        tma_load_2d(smem + Ly::kAhi + kb * kBlockBytes, tm_ahi, qa_full, kb * 64,
                                    ay);
                        tma_load_2d(smem + Ly::kAlo + kb * kBlockBytes, tm_alo, qa_full, kb * 64,
                                    ay);
                    }
                }
                ++qcount;
                for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                    const int s = (int)(tcount % kKSt);
                    const uint32_t par = (uint32_t)((tcount / kKSt) & 1) ^ 1u;
                    const int ky = (int)(U.kv_row0 + (long long)t * kTileKeys);
                    pf_step();
                    ok = in_range((long long)t * kTileKeys, U.n, A.status) &&
                         in_range(ky, kv_rows_total(P), A.status) &&
                         mbar_wait(&k_empty[s], par, abort_flag, P.wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&k_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kK + s * Ly::kOp + kb * kBlockBytes, tm_k,
                                    &k_full[s], kb * 64, ky);
                    ++kiss;
                    if constexpr (kX) {
                        const int sv = (int)(tcount % kVSt);
                        const uint32_t pv = (uint32_t)((tcount / kVSt) & 1) ^ 1u;
                        ok = mbar_wait(&v_empty[sv], pv, abort_flag, P.wait_ns);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&v_full[sv], Ly::kOp);
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb)
                            tma_load_2d(smem + Ly::kV + sv * Ly::kOp + kb * kBlockBytes, tm_v,
                                        &v_full[sv], kb * 64, ky);
                        ++viss;
                    }
                }
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            // drain: the last load issued into each buffer lands before the CTA exits
            // (the earlier ones were consumed before their buffer was refilled)
            if (qcount > 0) mbar_drain(qa_full, (uint32_t)((qcount - 1) & 1), kDrainNs);
            for (int s = 0; s < kKSt; ++s) {
                const long long ku = kiss / kKSt + ((kiss % kKSt) > s ? 1 : 0);
                if (ku > 0) mbar_drain(&k_full[s], (uint32_t)((ku - 1) & 1), kDrainNs);
            }
            for (int s = 0; s < kVSt; ++s) {
                const long long vu = viss / kVSt + ((viss % kVSt) > s ? 1 : 0);
                if (vu > 0) mbar_drain(&v_full[s], (uint32_t)((vu - 1) & 1), kDrainNs);
            }
        }
    } else if (run && warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            long long tcount = 0, icount = 0;
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, ncta, A, P, ord);
                const uint32_t idesc = idesc_bf16_f32(128, chunk_rows_n(P, it.c));
                ok = mbar_wait(qa_full, (uint32_t)(icount & 1), abort_flag, P.wait_ns);
                if (!ok) break;
                tc_fence_after();
                const uint64_t qb = sdesc_k_sw128(smem_u32(smem + Ly::kQ));
                const uint64_t hb = sdesc_k_sw128(smem_u32(smem + Ly::kAhi));
                const uint64_t lb = sdesc_k_sw128(smem_u32(smem + Ly::kAlo));
                for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                    const int s = (int)(tcount % kKSt);
                    const uint32_t par = (uint32_t)((tcount / kKSt) & 1);
                    const int b = (int)(tcount % kBufs);      // TMEM buffer of this tile
                    ok = mbar_wait(&tm_empty[b], (uint32_t)((tcount / kBufs) & 1) ^ 1u, abort_flag,
                                   P.wait_ns) &&
                         mbar_wait(&k_full[s], par, abort_flag, P.wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d_s = tmem + b * Ly::kBufCols;
                    const uint32_t d_x = d_s + 128;
                    const uint64_t ka = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
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
                    if constexpr (kX) {
                        const int sv = (int)(tcount % kVSt);
                        const uint32_t pv = (uint32_t)((tcount / kVSt) & 1);
                        ok = mbar_wait(&v_full[sv], pv, abort_flag, P.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t va = sdesc_k_sw128(smem_u32(smem + Ly::kV + sv * Ly::kOp));
                        mma_ss_c<false>(d_x, va, hb, idesc);
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t ko = kb * kBlockBytes + kk * 32;
                                if (kb | kk)
                                    mma_ss_c<true>(d_x, sdesc_add(va, ko), sdesc_add(hb, ko),
                                                   idesc);
                            }
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t ko = kb * kBlockBytes + kk * 32;
                                mma_ss_c<true>(d_x, sdesc_add(va, ko), sdesc_add(lb, ko), idesc);
                            }
                        mma_commit(&tm_full[b]);
                        mma_commit(&v_empty[sv]);
                    } else {
                        mma_commit(&tm_full[b]);
                    }
                }
                mma_commit(qa_empty);
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            // every MMA issued completes before TMEM is freed
            mma_commit(mma_done);
            mbar_drain(mma_done, 0, kDrainNs);
        }
    } else if (run && warp < 2 + kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;                  // TMEM lane quarter of this warp
        const int lane_base = quarter * 32 + ((warp - 2) >> 2) * 16;
        const int part = lane & 3;
        const int key0 = lane_base + (lane >> 2);      // tile-local keys: key0, key0 + 8
        const uint32_t lane_addr = (uint32_t)lane_base << 16;
        const float cscale = P.scale_log2;
        long long tcount = 0;
        bool ok = true;
        for (long long item = cta; ok && item < A.total_items; item += ncta) {
            const Item it = decode_item(item, ncta, A, P, ord);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int groups = chunk_rows_n(P, it.c) / 32;
            const int row_first = it.c * kChunkRows + 2 * part;   // unit-local row of pair 0
            // statistics of the thread's rows (pair rp: rows row_first + 8 rp + {0, 1})
            const float2 *u_ml = A.stat_ml + it.u * P.rows;
            const float *u_a2 = A.stat_a2 + it.u * P.rows;
            float2 nm[16], a2[16];
#pragma unroll
            for (int rp = 0; rp < 16; ++rp) {
                row_stats(u_ml, u_a2, row_first + 8 * rp, P.rows, nm[rp].x, a2[rp].x);
                row_stats(u_ml, u_a2, row_first + 8 * rp + 1, P.rows, nm[rp].y, a2[rp].y);
            }
            float *out = A.out + (long long)it.c * A.out_stride + U.kv_row0;
            const int pos0 = U.n - P.w;
            const float *u_v2 = A.v2 + U.kv_row0;
            float vq[2] = {0.f, 0.f};
            // the unit's rows of the score (or chunk partial) and ||v||^2 arrays
            const bool rows_ok =
                in_range(U.kv_row0, kv_rows_total(P), A.status) &&
                in_range(U.kv_row0 + U.n - 1, kv_rows_total(P), A.status) &&
                in_range(it.c, A.chunks, A.status);
            if constexpr (kX) {
                const int jf = it.t_begin * kTileKeys + key0;
                vq[0] = jf < U.n && rows_ok ? ld_v2<kCoherent>(u_v2 + jf) : 0.f;
                vq[1] = jf + 8 < U.n && rows_ok ? ld_v2<kCoherent>(u_v2 + jf + 8) : 0.f;
            }
            for (int t = it.t_begin; ok && t < it.t_end; ++t, ++tcount) {
                const int b = (int)(tcount % kBufs);          // TMEM buffer of this tile
                // ||v||^2 of the two keys of this tile (loaded a tile ahead)
                const float q0 = vq[0], q1 = vq[1];
                if (kX && t + 1 < it.t_end) {
                    const int jn = (t + 1) * kTileKeys + key0;
                    vq[0] = jn < U.n && rows_ok ? ld_v2<kCoherent>(u_v2 + jn) : 0.f;
                    vq[1] = jn + 8 < U.n && rows_ok ? ld_v2<kCoherent>(u_v2 + jn + 8) : 0.f;
                }
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&tm_full[b], (uint32_t)((tcount / kBufs) & 1), abort_flag,
                                          P.wait_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_col = tmem + lane_addr + b * Ly::kBufCols;
                const uint32_t x_col = s_col + 128;
                float sA[16], xA[16];
                const float2 v2[2] = {make_float2(q0, q0), make_float2(q1, q1)};
                const int j0 = t * kTileKeys + key0;
                const bool boundary = t * kTileKeys + kTileKeys - 1 > pos0;
                const int jrel[2] = {j0 - pos0, j0 + 8 - pos0};
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                if (!boundary) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (g < groups) {
                            tmem_ld16x256_x4(s_col + g * 32, sA);
                            if constexpr (kX) tmem_ld16x256_x4(x_col + g * 32, xA);
                            tmem_ld_wait();
                            reg_fence(sA);
                            if constexpr (kX) reg_fence(xA);
                            rescore_x4<RULE>(sA, xA, nm + 4 * g, a2 + 4 * g, cscale, v2, acc);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int g = 0; g < groups; ++g) {
                        tmem_ld16x256_x4(s_col + g * 32, sA);
                        if constexpr (kX) tmem_ld16x256_x4(x_col + g * 32, xA);
                        tmem_ld_wait();
                        reg_fence(sA);
                        if constexpr (kX) reg_fence(xA);
                        rescore_x4_window<RULE>(sA, xA, u_ml, u_a2, P.rows, row_first + 32 * g,
                                                P.w, jrel, cscale, v2, acc);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tm_empty[b]);
                float s0 = acc[0].x + acc[0].y, s1 = acc[1].x + acc[1].y;
                s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
                s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
                s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
                s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
                if (part == 0 && j0 < U.n && rows_ok) out[j0] = s0;
                if (part == 1 && j0 + 8 < U.n && rows_ok) out[j0 + 8] = s1;
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
    if (threadIdx.x == 0)
        for (int i = 0; i < Ly::kNumBars; ++i) mbar_inval(&bars[i]);
}

}  // namespace pass2
}  // namespace kvevict
