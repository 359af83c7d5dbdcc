// kv_pass1.cuh -- pass 1 of the DropKV score on the tcgen05 tensor cores:
// causal window attention over each unit's keys, split across CTAs (split-K),
// producing per split the row max m (log2 units), the row sum l of
// 2^(s*scale*log2 e - m) and the unnormalised output O = sum_j P_j v_j.  The
// merge in kv_score.cu combines the partials (DropKV, "Methodology in Plain
// English": the attention output a whose removal shift the score measures).
//
// Query-major.  A CTA runs two independent row sets ("lanes") over the key
// tiles of one split, each with its own S/P buffer and O accumulator in TMEM:
//   S_L = Q_L K^T    M = 128 rows, N = 128 keys, K = d   (fp32, TMEM cols 128 L)
//   O_L += P_L V     M = 128 rows, N = d, K = 128 keys   (fp32, TMEM cols 256 + 128 L;
//                    P is the A operand read from TMEM, V the MN-major B operand)
// When the unit's G*w window rows span two or more 128-row chunks, the lanes
// are two chunks sharing every K/V tile; with a single chunk, the lanes are the
// same rows over alternate tiles and each writes its own partial (the merge
// adds them like further splits).
//
// The MMA thread issues, per lane, P V of tile j and then S of tile j+1 into the
// same TMEM columns (the tensor pipe runs one thread's MMAs in order), so the
// softmax of one lane overlaps the MMAs of the other.  A softmax thread owns one
// row of its lane over all 128 keys of a tile: no exchange between threads.  It
// turns S into P' = 2^(s c - m + 13) and stores P' back over the S columns in
// fp16 (two keys per column).  P V runs in fp16: two converter warps turn each
// V tile in shared memory from bf16 to fp16 in place as it lands, which is exact for
// normal values below 65504 (larger ones post KV_ERR_UNSUPPORTED).  fp16 keeps
// 11 bits of p where bf16 keeps 8; a single bf16 P would leave a with ~2^-9
// relative error, which the rescoring expansion amplifies where a is close to
// a value row.  The running max is lazy: O and l are rescaled only when the
// tile max exceeds it by more than 2^2, so P' <= 2^15 stays in fp16 range and
// values down to 2^-37 p_max keep their mass.  l and O carry the factor 2^13,
// removed when the partial is written.  When S of tile j+1 is complete, P V of
// tile j is too, so the rescale needs no extra wait.
//
// The attention-sum rule needs only m and l: attn_stats_kernel (below) computes
// them from K alone.
//
// Warp roles (384 threads): warp 0 TMA producers (lane 0: the lanes' Q chunks per
// item and K tiles through a 3-stage ring; lane 1: V tiles through a 2- or
// 3-stage ring, each lane running as far ahead as its ring allows);
// warp 1 TMEM owner and MMA issuer; warps 2-5 softmax of lane 0, 6-9 of lane 1;
// warps 10-11 convert every V tile to fp16 as it lands (and compute ||v_j||^2),
// so neither lane's softmax waits for V or for the other lane.
// Work items are (unit, key split of up to 32768 keys, chunk pair), walked round-robin by a
// persistent grid.  All waits are bounded (KV_ERR_TIMEOUT on expiry).
//
// The passes are written as device bodies (attn_tc_body, attn_stats_body) that
// the stand-alone kernels in kv_attention.cu and the fused kernel in kv_fused.cu
// call with their CTA index and count.
#pragma once
#include <cfloat>

#include <cuda_fp16.h>

#include "kv_internal.cuh"
#include "kv_sm100.cuh"

namespace kvevict {
namespace pass1 {
using namespace sm100;

constexpr int kTileKeys = 128;
constexpr int kChunkRows = 128;
constexpr int kSoftWarps = 8;       // 4 per lane
constexpr int kConvWarps = 2;       // V tiles to fp16, ||v||^2
constexpr int kThreads = (2 + kSoftWarps + kConvWarps) * 32;
constexpr int kStatThreads = (2 + kSoftWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;     // O of lane L at column kOCol + 128 L
constexpr int kBlockBytes = 128 * 128;   // [128 rows][64 bf16], 128 B swizzle
constexpr float kRescaleLog2 = 2.f;
constexpr float kPScaleLog2 = 13.f;    // P' = p 2^13 in fp16

// Shared memory of attn_tc_body.  With two row chunks per item (chunk pairs) the
// CTA keeps both chunks' Q tiles, a 3-stage K ring and a 2-stage V ring.  With a
// single chunk (the lanes on alternate tiles; kOneQ) one Q tile serves both lanes
// and the second Q slot holds a third V stage.
template <int D, bool kOneQ = false>
struct Layout {
    static constexpr int kOp = (D / 64) * kBlockBytes;   // [128][D] bf16
    static constexpr int kQSlots = kOneQ ? 1 : 2;
    static constexpr int kKSt = 3;
    static constexpr int kVSt = kOneQ ? 3 : 2;
    static constexpr int kQ = 0;                          // Q of lane 0, then lane 1
    static constexpr int kK = kQ + kQSlots * kOp;
    static constexpr int kV = kK + kKSt * kOp;
    static constexpr int kBars = kV + kVSt * kOp;
    static constexpr int kNumBars = 2 * kKSt + 3 * kVSt + 2 + 4 * 2 + 1;
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kTotal = kMisc + 16;
};

struct AttnArgs {
    const int32_t *plan;       // [units + 1] prefix of key splits per unit
    float2 *part_ml;           // [units][max_splits * parts][rows]
    float *part_o;             // [units][max_splits * parts][rows][d]
    float *v2;                 // [L*H*N_tot] ||v_j||^2, written while converting V
    long long total_items;
    int pairs;                 // items per split: chunk pairs, or 1 with a single chunk
    int parts;                 // partials per split: 1 (chunk pairs) or 2 (alternate tiles)
    int chunks;
    int *status;
};

struct Item {
    long long u;
    int split, pair, t0, t1;   // tiles [t0, t1) of the split (unit-local tile index)
};

// `O` is the kernel's item-order parameter (used when O.nrun > 0).
__device__ __forceinline__ Item decode_item(long long item, const AttnArgs &A, const DevProblem &P,
                                            const ItemOrder &O) {
    Item it;
    it.pair = (int)(item % A.pairs);
    const long long gs = item / A.pairs;
    long long lo = 0;
    if (O.nrun > 0) {           // full splits first, then partial ones
        order_decode(O, gs, lo, it.split);
    } else {                    // many runs of lengths: the plan holds each unit's first split
        long long hi = P.units;
        while (hi - lo > 1) {
            const long long mid = (lo + hi) >> 1;
            if (A.plan[mid] <= gs) lo = mid; else hi = mid;
        }
        it.split = (int)(gs - A.plan[lo]);
    }
    it.u = lo;
    const int r = (int)(lo / ((long long)P.L * P.H));
    const int n = (int)(P.cu[r + 1] - P.cu[r]);
    const int k0 = it.split * P.split_keys;
    const int k1 = min(n, k0 + P.split_keys);
    it.t0 = k0 / kTileKeys;
    it.t1 = (k1 + kTileKeys - 1) / kTileKeys;
    return it;
}

// What lane L does in an item: `steps` tiles, the first at t0 + first, then
// every `stride` tiles; its rows are those of row chunk `chunk`.
struct LaneWork {
    int steps, first, stride, chunk;
};

__device__ __forceinline__ LaneWork lane_work(const AttnArgs &A, const Item &it, int L) {
    const int ntiles = it.t1 - it.t0;
    LaneWork w;
    if (A.parts == 1) {   // chunk pair sharing every tile
        w.chunk = 2 * it.pair + L;
        w.steps = w.chunk < A.chunks ? ntiles : 0;
        w.first = 0;
        w.stride = 1;
    } else {              // one chunk, alternate tiles
        w.chunk = 0;
        w.steps = (ntiles + 1 - L) / 2;
        w.first = L;
        w.stride = 2;
    }
    return w;
}

// Maximum of 32 values as a tree of 3-input maxima: depth 4 instead of a
// 16-long dependency chain.
__device__ __forceinline__ float max32_tree(const float (&v)[32]) {
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) a[i] = fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
    a[10] = fmaxf(v[30], v[31]);
    const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]);
    const float b2 = fmax3(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
    return fmaxf(fmax3(b0, b1, b2), b3);
}

// Two fp32 values as fp16x2 (round to nearest), the first in the low half.
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Two fp32 values as bf16x2 (round to nearest), the first in the low half.
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// P' of two keys as a bf16 pair: hi = bf16(p), lo = bf16(p - hi); hi + lo keeps 16
// bits of p (bf16 alone keeps 8, fp16 11).
__device__ __forceinline__ void split_bf162(float p0, float p1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf162(p0, p1);
    lo = pack_bf162(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xFFFF0000u));
}

// Masked form for tiles that reach the observation window: P' for 16 keys, zero
// for keys after `lim` (tile-local); adds P' to the row sum and stores the 8
// fp16x2 columns at `col`.
__device__ __forceinline__ void soft16_masked(const float *v, int j0, int lim, float cs,
                                              float negm, float2 &lsum, uint32_t col) {
    const float2 cs2 = make_float2(cs, cs);
    const float2 nm2 = make_float2(negm, negm);
    uint32_t w[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        const int j = 2 * h;
        const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), cs2, nm2);
        float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        if (j0 + j > lim) p.x = 0.f;
        if (j0 + j + 1 > lim) p.y = 0.f;
        lsum = __fadd2_rn(lsum, p);
        w[h] = pack_half2(p.x, p.y);
    }
    tmem_st8u(col, w);
}

// As soft16_masked with P' as a bf16 hi/lo pair: the 8 hi columns at `col`, the 8
// lo columns at `col` + 8 (the single-chunk layout of P in TMEM: per 16-key group
// q, hi at columns 16q .. 16q+7 and lo at 16q+8 .. 16q+15 of the S buffer).
__device__ __forceinline__ void soft16_masked_split(const float *v, int j0, int lim, float cs,
                                                    float negm, float2 &lsum, uint32_t col) {
    const float2 cs2 = make_float2(cs, cs);
    const float2 nm2 = make_float2(negm, negm);
    uint32_t w[16];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        const int j = 2 * h;
        const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), cs2, nm2);
        float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        if (j0 + j > lim) p.x = 0.f;
        if (j0 + j + 1 > lim) p.y = 0.f;
        lsum = __fadd2_rn(lsum, p);
        split_bf162(p.x, p.y, w[h], w[8 + h]);
    }
    tmem_st16u(col, w);
}

// Adds the squares of the two bf16 halves of `w` to `acc` (fp32 products of bf16
// are exact; one rounding per addition).
__device__ __forceinline__ void sq_acc_bf16x2(float &acc, uint32_t w) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.bf16 %0, lo, lo, %0;\n\tfma.rn.f32.bf16 %0, hi, hi, %0;\n\t}"
        : "+f"(acc)
        : "r"(w));
}

// Converts half of one key row of a swizzled [128][D] bf16 tile (`row`, 16-byte
// chunks [half * D/16, (half + 1) * D/16) across the 64-column blocks) to fp16 in
// place, and returns the sum of the squares of its bf16 values; `bad` is set if
// a value overflowed fp16.  `nz` collects the magnitude bits of the bf16 inputs
// and `nrm` the exponent bits of the fp16 outputs, so that the caller can tell
// a block of rows whose values are nonzero but all below fp16's normal range
// (2^-14), where fp16 keeps only a few of their bits.
template <int D>
__device__ __forceinline__ float row_half_to_f16(uint8_t *tile, int row, int half, bool &bad,
                                                 uint32_t &nz, uint32_t &nrm) {
    constexpr int kChunks = D / 16;            // 16-byte chunks per half row
    float acc[2] = {0.f, 0.f};
    uint32_t over = 0;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const int c = half * kChunks + i;      // logical chunk of the row
        uint4 *g = reinterpret_cast<uint4 *>(tile + (c >> 3) * kBlockBytes + row * 128 +
                                             (((c & 7) ^ (row & 7)) << 4));
        const uint4 w = *g;
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sq_acc_bf16x2(acc[k & 1], in[k]);
            o[k] = pack_half2(__uint_as_float(in[k] << 16), __uint_as_float(in[k] & 0xFFFF0000u));
            over |= ((o[k] & 0x7C00u) == 0x7C00u) | ((o[k] & 0x7C000000u) == 0x7C000000u);
            nz |= in[k] & 0x7FFF7FFFu;
            nrm |= o[k] & 0x7C007C00u;
        }
        *g = make_uint4(o[0], o[1], o[2], o[3]);
    }
    bad = bad || over != 0;
    return acc[0] + acc[1];
}

// Sum of the squares of the bf16 values of half of one key row of a swizzled
// [128][D] tile (as row_half_to_f16, without converting).
template <int D>
__device__ __forceinline__ float row_half_sq(const uint8_t *tile, int row, int half) {
    constexpr int kChunks = D / 16;
    float acc[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
        const int c = half * kChunks + i;
        const uint4 w = *reinterpret_cast<const uint4 *>(tile + (c >> 3) * kBlockBytes + row * 128 +
                                                         (((c & 7) ^ (row & 7)) << 4));
        sq_acc_bf16x2(acc[0], w.x);
        sq_acc_bf16x2(acc[1], w.y);
        sq_acc_bf16x2(acc[0], w.z);
        sq_acc_bf16x2(acc[1], w.w);
    }
    return acc[0] + acc[1];
}

// The kernel body, for CTA `cta` of `ncta` (all threads of the CTA call it;
// `tmem` is the base of 512 TMEM columns the caller allocated).  kOneQ selects the
// single-chunk form, for problems whose window rows fit one 128-row chunk
// (A.parts == 2; other problems post KV_ERR_UNSUPPORTED to it).  There the two
// lanes take alternate tiles and the tensor pipe has room to spare, while
// converting every V tile to fp16 would keep the two converter warps busy for
// most of a tile period (measured ~3600 of ~4000 clocks).  So V stays bf16 as it
// lands, P is written as a bf16 hi/lo pair (16 bits of p instead of fp16's 11)
// and P V runs as two MMA groups, P_hi V and P_lo V; the converter warps only
// compute ||v_j||^2.  V then has the whole bf16 range.
template <int D, bool kOneQ = false>
__device__ __forceinline__ void attn_tc_body(const DevProblem P, const CUtensorMap *tm_q,
                                             const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                             const AttnArgs A, const ItemOrder &ord, uint8_t *smem,
                                             uint32_t tmem, long long cta, long long ncta) {
    using Ly = Layout<D, kOneQ>;
    constexpr int kKStages = Ly::kKSt;
    constexpr int kVStages = Ly::kVSt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly::kBars);
    uint64_t *k_full = bars, *k_empty = bars + kKStages;
    uint64_t *v_full = bars + 2 * kKStages, *v_empty = v_full + kVStages;
    uint64_t *v_conv = v_empty + kVStages;  // [stage]: V tile converted to fp16 (2 warps)
    uint64_t *q_full = v_conv + kVStages, *q_empty = q_full + 1;
    uint64_t *s_full = q_empty + 1;        // [lane]: S of the lane's next tile is in TMEM
    uint64_t *p_full = s_full + 2;         // [lane]: P written (4 softmax warps)
    uint64_t *o_final = p_full + 2;        // [lane]: the lane's last P V of the item is done
    uint64_t *o_empty = o_final + 2;       // [lane]: O read out (4 softmax warps)
    uint64_t *mma_done = o_empty + 2;      // the MMA thread's last MMAs are done (exit)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Ly::kMisc + 4);

    if (threadIdx.x == 0) {
        *abort_flag = ((smem_u32(smem) & 1023u) || (kOneQ && A.parts != 2)) ? 1 : 0;
        if (*abort_flag) post_status(A.status, KV_ERR_UNSUPPORTED);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            // the last P V reading the stage frees it; in the single-chunk form the
            // converter warps, which then read the bf16 tile for ||v||^2 alongside
            // the MMAs, arrive too
            mbar_init(&v_empty[s], kOneQ ? 1 + kConvWarps : 1);
            mbar_init(&v_conv[s], kConvWarps);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int L = 0; L < 2; ++L) {
            mbar_init(&s_full[L], 1);
            mbar_init(&p_full[L], kSoftWarps / 2);
            mbar_init(&o_final[L], 1);
            mbar_init(&o_empty[L], kSoftWarps / 2);
        }
        mbar_init(mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(tm_q);
        prefetch_tensormap(tm_k);
        prefetch_tensormap(tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool run = *abort_flag == 0;

    if (run && warp == 0) {
        // ------------------------------------------------------------ producers
        // Lane 0 loads each item's Q and the K tiles, lane 1 the V tiles, each as
        // far ahead as its own ring allows: a V tile is requested as soon as its
        // stage frees, not after the K tiles before it (its HBM latency then hides
        // behind the tiles in flight).
        if (lane == 0) {
            long long tcount = 0, icount = 0;   // K tiles loaded, items
            long long qcount = 0, kiss = 0;     // Q and K loads issued
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, A, P, ord);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                const LaneWork w0 = lane_work(A, it, 0), w1 = lane_work(A, it, 1);
                const bool two_q = A.parts == 1 && w1.steps > 0;
                ok = mbar_wait(q_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, P.wait_ns);
                if (!ok) break;
                mbar_arrive_expect_tx(q_full, (two_q ? 2 : 1) * Ly::kOp);
                for (int L = 0; L < (two_q ? 2 : 1); ++L) {
                    const int qy = (int)(U.q_row0 + (L ? w1.chunk : w0.chunk) * kChunkRows);
                    if (!in_range(qy, q_rows_total(P), A.status)) ok = false;
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kQ + L * Ly::kOp + kb * kBlockBytes, tm_q,
                                    q_full, kb * 64, qy);
                }
                ++qcount;
                const int ntiles = it.t1 - it.t0;
                for (int i = 0; ok && i < ntiles; ++i) {
                    const long long kc = tcount + i;
                    const int s = (int)(kc % kKStages);
                    const int ky = (int)(U.kv_row0 + (long long)(it.t0 + i) * kTileKeys);
                    ok = in_range((it.t0 + i) * kTileKeys, U.n, A.status) &&
                         in_range(ky, kv_rows_total(P), A.status) &&
                         mbar_wait(&k_empty[s], (uint32_t)((kc / kKStages) & 1) ^ 1u, abort_flag,
                                   P.wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&k_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kK + s * Ly::kOp + kb * kBlockBytes, tm_k,
                                    &k_full[s], kb * 64, ky);
                    ++kiss;
                }
                tcount += ntiles;
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            // drain: the last load issued into each buffer lands before the CTA exits
            // (the earlier ones were consumed before their buffer was refilled)
            if (qcount > 0) mbar_drain(q_full, (uint32_t)((qcount - 1) & 1), kDrainNs);
            for (int s = 0; s < kKStages; ++s) {
                const long long uses = kiss / kKStages + ((kiss % kKStages) > s ? 1 : 0);
                if (uses > 0) mbar_drain(&k_full[s], (uint32_t)((uses - 1) & 1), kDrainNs);
            }
        } else if (lane == 1) {
            long long tcount = 0, viss = 0;     // V tiles loaded (= issued)
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, A, P, ord);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                const int ntiles = it.t1 - it.t0;
                for (int i = 0; ok && i < ntiles; ++i) {
                    const long long vc = tcount + i;
                    const int s = (int)(vc % kVStages);
                    const int vy = (int)(U.kv_row0 + (long long)(it.t0 + i) * kTileKeys);
                    ok = in_range((it.t0 + i) * kTileKeys, U.n, A.status) &&
                         in_range(vy, kv_rows_total(P), A.status) &&
                         mbar_wait(&v_empty[s], (uint32_t)((vc / kVStages) & 1) ^ 1u, abort_flag,
                                   P.wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&v_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kV + s * Ly::kOp + kb * kBlockBytes, tm_v,
                                    &v_full[s], kb * 64, vy);
                    ++viss;
                }
                tcount += ntiles;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            for (int s = 0; s < kVStages; ++s) {
                const long long uses = viss / kVStages + ((viss % kVStages) > s ? 1 : 0);
                if (uses > 0) mbar_drain(&v_full[s], (uint32_t)((uses - 1) & 1), kDrainNs);
            }
        }
    } else if (run && warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(128, kTileKeys);
            const uint32_t idesc_pv = idesc_f16_f32_bmn(128, D);
            const uint32_t idesc_pv_bf = idesc_bf16_f32_bmn(128, D);
            long long tcount = 0, icount = 0;
            long long sc[2] = {0, 0};   // steps issued per lane
            long long oc[2] = {0, 0};   // items in which the lane took part
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, A, P, ord);
                const LaneWork w[2] = {lane_work(A, it, 0), lane_work(A, it, 1)};
                // the lane whose MMAs are the last to read a tile frees its K/V stage
                const int releaser = (A.parts == 1 && w[1].steps > 0) ? 1 : -1;
                ok = mbar_wait(q_full, (uint32_t)(icount & 1), abort_flag, P.wait_ns);
                if (!ok) break;
                tc_fence_after();
                auto frees = [&](int L) { return releaser < 0 || releaser == L; };
                // S_L = Q_L K^T for step j of lane L
                auto issue_s = [&](int L, int j) {
                    const long long kc = tcount + w[L].first + (long long)j * w[L].stride;
                    const int s = (int)(kc % kKStages);
                    ok = ok && mbar_wait(&k_full[s], (uint32_t)((kc / kKStages) & 1), abort_flag,
                                         P.wait_ns);
                    if (!ok) return;
                    tc_fence_after();
                    const uint64_t qa = sdesc_k_sw128(
                        smem_u32(smem + Ly::kQ + (A.parts == 1 ? L : 0) * Ly::kOp));
                    const uint64_t kb0 = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
                    const uint32_t d_s = tmem + 128 * L;
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t ko = kb * kBlockBytes + kk * 32;
                            if (kb | kk)
                                mma_ss_c<true>(d_s, sdesc_add(qa, ko), sdesc_add(kb0, ko), idesc_s);
                            else
                                mma_ss_c<false>(d_s, qa, kb0, idesc_s);
                        }
                    mma_commit(&s_full[L]);
                    if (frees(L)) mma_commit(&k_empty[s]);
                };
                // O_L (+)= P' V for step j of lane L (fp16 operands)
                auto issue_pv = [&](int L, int j) {
                    const long long vc = tcount + w[L].first + (long long)j * w[L].stride;
                    const int s = (int)(vc % kVStages);
                    if (j == 0)
                        ok = ok && mbar_wait(&o_empty[L], (uint32_t)(oc[L] & 1) ^ 1u, abort_flag,
                                             P.wait_ns);
                    ok = ok && mbar_wait(&p_full[L], (uint32_t)((sc[L] + j) & 1), abort_flag,
                                         P.wait_ns);
                    // the single-chunk form multiplies the bf16 tile as it landed; the
                    // other waits for its conversion to fp16
                    ok = ok && mbar_wait(kOneQ ? &v_full[s] : &v_conv[s],
                                         (uint32_t)((vc / kVStages) & 1), abort_flag, P.wait_ns);
                    if (!ok) return;
                    tc_fence_after();
                    const uint64_t vb =
                        sdesc_mn_sw128(smem_u32(smem + Ly::kV + s * Ly::kOp), kBlockBytes);
                    const uint32_t pcol = tmem + 128 * L;
                    const uint32_t d_o = tmem + kOCol + 128 * L;
#pragma unroll
                    for (int q = 0; q < kTileKeys / 16; ++q) {
                        const uint64_t bd = sdesc_add(vb, q * 16 * 128);
                        if constexpr (kOneQ) {
                            // keys 16q..16q+15: P_hi in bf16x2 columns 16q..16q+7, P_lo in
                            // 16q+8..16q+15
                            const uint32_t a = pcol + q * 16;
                            if (j == 0 && q == 0)
                                mma_ts_c<false>(d_o, a, bd, idesc_pv_bf);
                            else
                                mma_ts_c<true>(d_o, a, bd, idesc_pv_bf);
                            mma_ts_c<true>(d_o, a + 8, bd, idesc_pv_bf);
                        } else {
                            // keys 16q..16q+15: fp16x2 columns 8q..8q+7
                            const uint32_t a = pcol + q * 8;
                            if (j == 0 && q == 0)
                                mma_ts_c<false>(d_o, a, bd, idesc_pv);
                            else
                                mma_ts_c<true>(d_o, a, bd, idesc_pv);
                        }
                    }
                    if (frees(L)) mma_commit(&v_empty[s]);
                };
                const int nmax = max(w[0].steps, w[1].steps);
                for (int L = 0; L < 2; ++L)
                    if (w[L].steps > 0) issue_s(L, 0);
                for (int j = 0; ok && j < nmax; ++j)
                    for (int L = 0; ok && L < 2; ++L)
                        if (j < w[L].steps) {
                            issue_pv(L, j);
                            if (j + 1 < w[L].steps) issue_s(L, j + 1);
                            if (ok && j + 1 == w[L].steps) mma_commit(&o_final[L]);
                        }
                mma_commit(q_empty);
                for (int L = 0; L < 2; ++L) {
                    sc[L] += w[L].steps;
                    if (w[L].steps > 0) ++oc[L];
                }
                tcount += it.t1 - it.t0;
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
    } else if (run && warp < 2 + kSoftWarps) {
        // ------------------------------------------------------------ softmax
        const int L = (warp - 2) >> 2;                    // lane (row set) of this warp
        const int quarter = warp & 3;
        const int rr = quarter * 32 + lane;               // row of the chunk = TMEM lane
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_base = tmem + lane_addr + 128 * L;
        const uint32_t o_base = tmem + lane_addr + kOCol + 128 * L;
        const float cs = P.scale_log2;
        long long sc = 0, oc = 0;
        bool ok = true;
        for (long long item = cta; ok && item < A.total_items; item += ncta) {
            const Item it = decode_item(item, A, P, ord);
            const LaneWork w = lane_work(A, it, L);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int row = w.chunk * kChunkRows + rr;
            const int slot = A.parts == 1 ? it.split : 2 * it.split + L;
            const size_t prow_idx =
                ((size_t)it.u * P.max_splits * A.parts + slot) * P.rows + row;
            const bool row_valid =
                row < P.rows &&
                in_range((long long)prow_idx, P.units * P.max_splits * A.parts * P.rows, A.status);
            if (w.steps == 0) {
                // no tile for this lane: an empty partial (l = 0) for the merge to skip
                if (A.parts == 2 && row_valid) A.part_ml[prow_idx] = make_float2(-INFINITY, 0.f);
                continue;
            }
            const int pos = U.n - P.w + (row % P.w);      // last key this row sees
            const int pos_min = U.n - P.w;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; ok && j < w.steps; ++j) {
                const int ti = w.first + j * w.stride;
                const int kt = (it.t0 + ti) * kTileKeys;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[L], (uint32_t)((sc + j) & 1),
                                                       abort_flag, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
                // only tiles that reach into the window need the causal mask
                const bool boundary = kt + kTileKeys - 1 > pos_min;
                const int lim = row_valid ? pos - kt : -1;
                float mx = -INFINITY;
                if (!boundary) {
                    float sa[32], sb[32];
                    tmem_ld32(s_base, sa);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float(&cur)[32] = (c & 1) ? sb : sa;
                        float(&nxt)[32] = (c & 1) ? sa : sb;
                        tmem_ld_wait();
                        reg_fence(cur);
                        if (c < 3) tmem_ld32(s_base + 32 * (c + 1), nxt);
                        mx = fmaxf(mx, max32_tree(cur));
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < kTileKeys / 16; ++c) {
                        float sv[16];
                        tmem_ld16(s_base + 16 * c, sv);
                        tmem_ld_wait();
                        reg_fence(sv);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            mx = fmaxf(mx, 16 * c + i > lim ? -INFINITY : sv[i]);
                    }
                }
                const float m_tile = mx * cs;
                const bool need = m_tile > m_used + kRescaleLog2;
                const float factor = need ? ex2_approx(m_used - m_tile) : 1.f;
                if (__any_sync(0xffffffffu, need && j > 0)) {
                    // O_L holds P V of the earlier tiles; that P V is complete (S of
                    // this tile was issued after it), so rescale it in place
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(o_base + 32 * c, o);
                        tmem_ld_wait();
                        reg_fence(o);
                        uint32_t ou[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) ou[i] = __float_as_uint(o[i] * factor);
                        tmem_st32u(o_base + 32 * c, ou);
                    }
                }
                if (need) {
                    l *= factor;
                    m_used = m_tile;
                }
                // P' = 2^(s c - m + 13); with m = -inf (every key masked so far) p = 0
                const float negm = m_used == -INFINITY ? 0.f : kPScaleLog2 - m_used;
                float2 lsum = make_float2(0.f, 0.f);
                if (!boundary) {
                    const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(negm, negm);
                    float sa[32], sb[32];
                    tmem_ld32(s_base, sa);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float(&cur)[32] = (c & 1) ? sb : sa;
                        float(&nxt)[32] = (c & 1) ? sa : sb;
                        tmem_ld_wait();
                        reg_fence(cur);
                        if (c < 3) tmem_ld32(s_base + 32 * (c + 1), nxt);
                        // keys 32c..32c+31 -> fp16x2 columns 16c..16c+15, or in the
                        // single-chunk form bf16x2 hi/lo columns 32c..32c+31: only
                        // columns of keys already read are overwritten
                        uint32_t pw[kOneQ ? 32 : 16];
                        float2 ps[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                        make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 t = __ffma2_rn(make_float2(cur[i], cur[i + 1]), cs2, nm2);
                            const float p0 = ex2_approx(t.x), p1 = ex2_approx(t.y);
                            ps[(i / 2) & 3] = __fadd2_rn(ps[(i / 2) & 3], make_float2(p0, p1));
                            if constexpr (kOneQ)
                                split_bf162(p0, p1, pw[(i / 16) * 16 + (i % 16) / 2],
                                            pw[(i / 16) * 16 + 8 + (i % 16) / 2]);
                            else
                                pw[i / 2] = pack_half2(p0, p1);
                        }
                        if constexpr (kOneQ)
                            tmem_st32u(s_base + 32 * c, pw);
                        else
                            tmem_st16u(s_base + 16 * c, pw);
                        lsum = __fadd2_rn(lsum, __fadd2_rn(__fadd2_rn(ps[0], ps[1]),
                                                           __fadd2_rn(ps[2], ps[3])));
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < kTileKeys / 16; ++c) {
                        float sv[16];
                        tmem_ld16(s_base + 16 * c, sv);
                        tmem_ld_wait();
                        reg_fence(sv);
                        if constexpr (kOneQ)
                            soft16_masked_split(sv, 16 * c, lim, cs, negm, lsum, s_base + 16 * c);
                        else
                            soft16_masked(sv, 16 * c, lim, cs, negm, lsum, s_base + 8 * c);
                    }
                }
                l += lsum.x + lsum.y;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[L]);
            }
            if (!ok) break;
            // item end: read O_L once the lane's last P V is done, write the partial
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&o_final[L], (uint32_t)(oc & 1), abort_flag, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            // O and l carry P's factor 2^13; the partial is written without it
            constexpr float kUnscale = 1.f / 8192.f;
            float *po = A.part_o + prow_idx * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(o_base + 32 * c, o);
                tmem_ld_wait();
                reg_fence(o);
                if (row_valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(po + 32 * c + i) =
                            make_float4(o[i] * kUnscale, o[i + 1] * kUnscale,
                                        o[i + 2] * kUnscale, o[i + 3] * kUnscale);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[L]);
            if (row_valid) A.part_ml[prow_idx] = make_float2(m_used, l * kUnscale);
            sc += w.steps;
            ++oc;
        }
        if (!ok) {
            *abort_flag = 1;
            post_status(A.status, KV_ERR_TIMEOUT);
        }
    } else if (run) {
        // ------------------------------------------------------------ V conversion
        // Every V tile of the item, in load order: warp cw converts rows 64 cw ..
        // 64 cw + 63 to fp16 in place, two threads per row (lane, lane ^ 16), and
        // writes ||v_j||^2 of those keys for the rescoring pass.
        const int cw = warp - 2 - kSoftWarps;
        long long tbase = 0;   // tiles of this CTA's earlier items (V stage and parity)
        bool ok = true;
        for (long long item = cta; ok && item < A.total_items; item += ncta) {
            const Item it = decode_item(item, A, P, ord);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int item_tiles = it.t1 - it.t0;
            for (int ti = 0; ok && ti < item_tiles; ++ti) {
                const long long vc = tbase + ti;
                const int s = (int)(vc % kVStages);
                ok = __all_sync(0xffffffffu, mbar_wait(&v_full[s], (uint32_t)((vc / kVStages) & 1),
                                                       abort_flag, P.wait_ns));
                if (!ok) break;
                uint8_t *tile = smem + Ly::kV + s * Ly::kOp;
                if constexpr (kOneQ) {
                    // ||v||^2 of the bf16 tile, read alongside the MMAs; then this
                    // warp's share of the stage's release
#pragma unroll 1
                    for (int k0 = 0; k0 < 64; k0 += 16) {
                        const int row = cw * 64 + k0 + (lane & 15);
                        float q = row_half_sq<D>(tile, row, lane >> 4);
                        q += __shfl_xor_sync(0xffffffffu, q, 16);
                        const int j = (it.t0 + ti) * kTileKeys + row;
                        if (lane < 16 && j < U.n &&
                            in_range(U.kv_row0 + j, kv_rows_total(P), A.status))
                            A.v2[U.kv_row0 + j] = q;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&v_empty[s]);
                    continue;
                }
                bool bad = false;
                uint32_t nz = 0, nrm = 0;
#pragma unroll 1
                for (int k0 = 0; k0 < 64; k0 += 16) {
                    const int row = cw * 64 + k0 + (lane & 15);
                    float q = row_half_to_f16<D>(tile, row, lane >> 4, bad, nz, nrm);
                    q += __shfl_xor_sync(0xffffffffu, q, 16);
                    const int j = (it.t0 + ti) * kTileKeys + row;   // key of the unit
                    if (lane < 16 && j < U.n &&
                        in_range(U.kv_row0 + j, kv_rows_total(P), A.status))
                        A.v2[U.kv_row0 + j] = q;
                }
                // refused: a value fp16 cannot hold, or 64 rows of nonzero values that
                // all fall below 2^-14 (fp16 subnormals keep too few of their bits)
                const bool tiny = __any_sync(0xffffffffu, nz != 0) &&
                                  !__any_sync(0xffffffffu, nrm != 0);
                if (bad || (tiny && lane == 0)) post_status(A.status, KV_ERR_UNSUPPORTED);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&v_conv[s]);
            }
            tbase += item_tiles;
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

// ---------------------------------------------------------------------------
// Row statistics only (score rule KV_SCORE_ATTN_SUM).  The attention sum needs
// per window row just m and l (PyramidKV guide, "Observation Window and
// Aggregated Attention Eviction": S_j sums the softmax weights, which need the
// row's normaliser and nothing else), so this pass streams K alone: per tile
// S_L = Q_L K^T into one of two TMEM buffers of lane L, and the softmax warps
// keep a running (m, l) per row with one ex2 per (row, key).  Same items,
// lanes and partial layout as attn_tc_kernel; the merge reads only (m, l).
// Warp roles: warp 0 producer (Q per item, K through a 4-stage ring), warp 1
// TMEM owner and MMA issuer, warps 2-5 rows of lane 0, 6-9 rows of lane 1.
// ---------------------------------------------------------------------------
constexpr int kStatKSt = 4;
constexpr float kStatLazyLog2 = 8.f;   // m is raised only when a chunk max exceeds it by 2^8

template <int D>
struct StatLayout {
    static constexpr int kOp = (D / 64) * kBlockBytes;
    static constexpr int kQ = 0;                          // Q of lane 0, then lane 1
    static constexpr int kK = kQ + 2 * kOp;
    static constexpr int kBars = kK + kStatKSt * kOp;
    static constexpr int kNumBars = 2 * kStatKSt + 2 + 4 + 4 + 1;
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kTotal = kMisc + 16;
};

// The kernel body, called as attn_tc_body is; warps from 2 + kSoftWarps on idle.
template <int D>
__device__ __forceinline__ void attn_stats_body(const DevProblem P, const CUtensorMap *tm_q,
                                                const CUtensorMap *tm_k, const AttnArgs A,
                                                const ItemOrder &ord, uint8_t *smem, uint32_t tmem,
                                                long long cta, long long ncta) {
    using Ly = StatLayout<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly::kBars);
    uint64_t *k_full = bars, *k_empty = bars + kStatKSt;
    uint64_t *q_full = bars + 2 * kStatKSt, *q_empty = q_full + 1;
    uint64_t *s_full = q_empty + 1;        // [2 L + b]: S in buffer b of lane L
    uint64_t *s_free = s_full + 4;         // [2 L + b]: buffer read (4 warps)
    uint64_t *mma_done = s_free + 4;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Ly::kMisc + 4);

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort_flag) post_status(A.status, KV_ERR_UNSUPPORTED);
        for (int s = 0; s < kStatKSt; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < 4; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], kSoftWarps / 2);
        }
        mbar_init(mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(tm_q);
        prefetch_tensormap(tm_k);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool run = *abort_flag == 0;


    if (run && warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            long long tcount = 0, icount = 0, qcount = 0, kiss = 0;
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, A, P, ord);
                const UnitInfo U = unit_info(P, it.u, P.cu);
                const LaneWork w0 = lane_work(A, it, 0), w1 = lane_work(A, it, 1);
                const bool two_q = A.parts == 1 && w1.steps > 0;
                ok = mbar_wait(q_empty, (uint32_t)(icount & 1) ^ 1u, abort_flag, P.wait_ns);
                if (!ok) break;
                mbar_arrive_expect_tx(q_full, (two_q ? 2 : 1) * Ly::kOp);
                for (int L = 0; L < (two_q ? 2 : 1); ++L) {
                    const int qy = (int)(U.q_row0 + (L ? w1.chunk : w0.chunk) * kChunkRows);
                    if (!in_range(qy, q_rows_total(P), A.status)) ok = false;
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kQ + L * Ly::kOp + kb * kBlockBytes, tm_q,
                                    q_full, kb * 64, qy);
                }
                ++qcount;
                const int ntiles = it.t1 - it.t0;
                for (int i = 0; ok && i < ntiles; ++i) {
                    const long long kc = tcount + i;
                    const int s = (int)(kc % kStatKSt);
                    const int ky = (int)(U.kv_row0 + (long long)(it.t0 + i) * kTileKeys);
                    ok = in_range((it.t0 + i) * kTileKeys, U.n, A.status) &&
                         in_range(ky, kv_rows_total(P), A.status) &&
                         mbar_wait(&k_empty[s], (uint32_t)((kc / kStatKSt) & 1) ^ 1u, abort_flag,
                                   P.wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&k_full[s], Ly::kOp);
#pragma unroll
                    for (int kb = 0; kb < D / 64; ++kb)
                        tma_load_2d(smem + Ly::kK + s * Ly::kOp + kb * kBlockBytes, tm_k,
                                    &k_full[s], kb * 64, ky);
                    ++kiss;
                }
                tcount += ntiles;
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            if (qcount > 0) mbar_drain(q_full, (uint32_t)((qcount - 1) & 1), kDrainNs);
            for (int s = 0; s < kStatKSt; ++s) {
                const long long uses = kiss / kStatKSt + ((kiss % kStatKSt) > s ? 1 : 0);
                if (uses > 0) mbar_drain(&k_full[s], (uint32_t)((uses - 1) & 1), kDrainNs);
            }
        }
    } else if (run && warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(128, kTileKeys);
            long long tcount = 0, icount = 0;
            long long sc[2] = {0, 0};   // S tiles issued per lane (buffer and parity)
            bool ok = true;
            for (long long item = cta; ok && item < A.total_items; item += ncta) {
                const Item it = decode_item(item, A, P, ord);
                const LaneWork w[2] = {lane_work(A, it, 0), lane_work(A, it, 1)};
                const int releaser = (A.parts == 1 && w[1].steps > 0) ? 1 : -1;
                ok = mbar_wait(q_full, (uint32_t)(icount & 1), abort_flag, P.wait_ns);
                if (!ok) break;
                tc_fence_after();
                const int nmax = max(w[0].steps, w[1].steps);
                for (int j = 0; ok && j < nmax; ++j)
                    for (int L = 0; ok && L < 2; ++L) {
                        if (j >= w[L].steps) continue;
                        const long long cnt = sc[L] + j;
                        const int b = (int)(cnt & 1);
                        const long long kc = tcount + w[L].first + (long long)j * w[L].stride;
                        const int s = (int)(kc % kStatKSt);
                        ok = mbar_wait(&s_free[2 * L + b], (uint32_t)((cnt >> 1) & 1) ^ 1u,
                                       abort_flag, P.wait_ns) &&
                             mbar_wait(&k_full[s], (uint32_t)((kc / kStatKSt) & 1), abort_flag,
                                       P.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t qa = sdesc_k_sw128(
                            smem_u32(smem + Ly::kQ + (A.parts == 1 ? L : 0) * Ly::kOp));
                        const uint64_t kb0 = sdesc_k_sw128(smem_u32(smem + Ly::kK + s * Ly::kOp));
                        const uint32_t d_s = tmem + 256 * L + 128 * b;
#pragma unroll
                        for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint32_t ko = kb * kBlockBytes + kk * 32;
                                if (kb | kk)
                                    mma_ss_c<true>(d_s, sdesc_add(qa, ko), sdesc_add(kb0, ko),
                                                   idesc_s);
                                else
                                    mma_ss_c<false>(d_s, qa, kb0, idesc_s);
                            }
                        mma_commit(&s_full[2 * L + b]);
                        if (releaser < 0 || releaser == L) mma_commit(&k_empty[s]);
                    }
                mma_commit(q_empty);
                sc[0] += w[0].steps;
                sc[1] += w[1].steps;
                tcount += it.t1 - it.t0;
                ++icount;
            }
            if (!ok) {
                *abort_flag = 1;
                post_status(A.status, KV_ERR_TIMEOUT);
            }
            mma_commit(mma_done);
            mbar_drain(mma_done, 0, kDrainNs);
        }
    } else if (run && warp < 2 + kSoftWarps) {
        // ------------------------------------------------------------ row statistics
        const int L = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int rr = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float cs = P.scale_log2;
        const float2 cs2 = make_float2(cs, cs);
        long long sc = 0;
        bool ok = true;
        for (long long item = cta; ok && item < A.total_items; item += ncta) {
            const Item it = decode_item(item, A, P, ord);
            const LaneWork w = lane_work(A, it, L);
            const UnitInfo U = unit_info(P, it.u, P.cu);
            const int row = w.chunk * kChunkRows + rr;
            const int slot = A.parts == 1 ? it.split : 2 * it.split + L;
            const size_t prow_idx =
                ((size_t)it.u * P.max_splits * A.parts + slot) * P.rows + row;
            const bool row_valid =
                row < P.rows &&
                in_range((long long)prow_idx, P.units * P.max_splits * A.parts * P.rows, A.status);
            if (w.steps == 0) {
                if (A.parts == 2 && row_valid) A.part_ml[prow_idx] = make_float2(-INFINITY, 0.f);
                continue;
            }
            const int pos = U.n - P.w + (row % P.w);
            const int pos_min = U.n - P.w;
            float m = -INFINITY, l = 0.f;
            // one 32-key chunk: raise m lazily, then l += sum of 2^(s c - m)
            auto chunk32 = [&](const float (&v)[32]) {
                const float mt = max32_tree(v) * cs;
                const bool up = mt > m + kStatLazyLog2;
                l *= up ? ex2_approx(m - mt) : 1.f;
                m = up ? mt : m;
                const float2 nm2 = make_float2(-m, -m);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float2 t = __ffma2_rn(make_float2(v[i], v[i + 1]), cs2, nm2);
                    acc[(i / 2) & 3] = __fadd2_rn(acc[(i / 2) & 3],
                                                  make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                }
                const float2 a01 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                l += a01.x + a01.y;
            };
            for (int j = 0; ok && j < w.steps; ++j) {
                const int ti = w.first + j * w.stride;
                const int kt = (it.t0 + ti) * kTileKeys;
                const long long cnt = sc + j;
                const int b = (int)(cnt & 1);
                ok = __all_sync(0xffffffffu, mbar_wait(&s_full[2 * L + b],
                                                       (uint32_t)((cnt >> 1) & 1), abort_flag,
                                                       P.wait_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_base = tmem + lane_addr + 256 * L + 128 * b;
                if (kt + kTileKeys - 1 <= pos_min) {
                    // every row of the chunk sees every key of the tile
                    float sa[32], sb[32];
                    tmem_ld32(s_base, sa);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float(&cur)[32] = (c & 1) ? sb : sa;
                        float(&nxt)[32] = (c & 1) ? sa : sb;
                        tmem_ld_wait();
                        reg_fence(cur);
                        if (c < 3) {
                            tmem_ld32(s_base + 32 * (c + 1), nxt);
                        } else {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&s_free[2 * L + b]);
                        }
                        chunk32(cur);
                    }
                } else {
                    // the tile reaches the window: key kt + i is seen when i <= lim
                    const int lim = row_valid ? pos - kt : -1;
#pragma unroll 1
                    for (int c = 0; c < kTileKeys / 16; ++c) {
                        float sv[16];
                        tmem_ld16(s_base + 16 * c, sv);
                        tmem_ld_wait();
                        reg_fence(sv);
                        if (c == kTileKeys / 16 - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&s_free[2 * L + b]);
                        }
                        float mx = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            mx = fmaxf(mx, 16 * c + i > lim ? -INFINITY : sv[i]);
                        const float mt = mx * cs;
                        const bool up = mt > m + kStatLazyLog2;
                        l *= up ? ex2_approx(m - mt) : 1.f;
                        m = up ? mt : m;
                        float acc = 0.f;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc += 16 * c + i > lim ? 0.f : ex2_approx(fmaf(sv[i], cs, -m));
                        l += acc;
                    }
                }
            }
            if (!ok) break;
            if (row_valid) A.part_ml[prow_idx] = make_float2(m, l);
            sc += w.steps;
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

}  // namespace pass1
}  // namespace kvevict
