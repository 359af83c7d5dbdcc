// kv_compact.cuh -- ragged gather of the kept K/V rows into one packed cache.
//
// Output row i of unit u (offsets[u] <= i < offsets[u+1]) is the K (and V)
// row of token sel[i] of that unit: a bit copy (GraceKV, "physical cache
// packing": one cache of its own length per layer-KV-head).  Each CTA copies a
// contiguous range of output rows, finding each row's unit by binary search in
// the offsets table between the units of its first and last rows; a warp moves one
// row pair (K and V) per step in 16-byte vectors, four rows in flight, with
// read-only loads and streaming stores (the copy is touched once).
//
// Block form (BellowsKV blog, eviction operator: one decision per block of
// consecutive layers): unit (r, l, h) takes its indices from the selection of
// block unit (r, l / block_layers), row i of the unit reading index i of the
// block's list.
//
// compact_block is the device function the stand-alone kernels (kv_compact.cu)
// and the fused kernel (kv_fused.cu) call per block of output rows.
#pragma once
#include "kv_internal.cuh"

namespace kvevict {

constexpr int kRowsPerCta = 256;   // output rows one compact_block call copies

__device__ __forceinline__ uint4 ld_nc(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_cs(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Where a unit's indices come from in the block form.
struct BlockSel {
    const int32_t *sel;        // indices of the block units
    const int64_t *offsets;    // [R * nblk + 1] offsets of the block units
    int block_layers;          // 0: the plain form
    int nblk;                  // L / block_layers
};

// Copies output rows [blk * kRowsPerCta, +kRowsPerCta) with the kWarps warps of
// the calling CTA (all call it), kUnroll rows in flight per warp.  s_unit and
// s_range are kRowsPerCta + 2 words of shared memory.
template <int D, int kWarps, int kUnroll>
__device__ __forceinline__ void compact_block(const DevProblem &P, const uint4 *__restrict__ k,
                                              const uint4 *__restrict__ v,
                                              const int32_t *__restrict__ sel,
                                              const int64_t *__restrict__ offsets,
                                              long long total_rows, uint4 *__restrict__ kout,
                                              uint4 *__restrict__ vout, const BlockSel &B,
                                              long long blk, long long *s_unit,
                                              long long *s_range) {
    constexpr int CPR = D / 8;                    // 16-byte chunks per row
    constexpr int LANES = 2 * CPR;                // K chunks then V chunks
    constexpr int ROWS_PER_PASS = 32 / LANES;     // rows one warp covers per step
    static_assert(32 % LANES == 0, "row must split evenly over a warp");
    const long long row0 = blk * kRowsPerCta;
    const long long left = total_rows - row0;
    const int nrows = (int)(left < kRowsPerCta ? left : kRowsPerCta);
    if (nrows <= 0) return;
    auto unit_of = [&](long long row, long long lo, long long hi) {   // offsets[lo] <= row < offsets[hi]
        while (hi - lo > 1) {
            const long long mid = (lo + hi) >> 1;
            if (offsets[mid] <= row) lo = mid; else hi = mid;
        }
        return lo;
    };
    // units of the first and last rows, then of every row within that range
    if (threadIdx.x < 2)
        s_range[threadIdx.x] = unit_of(row0 + (threadIdx.x ? nrows - 1 : 0), 0, P.units);
    __syncthreads();
    for (int i = threadIdx.x; i < nrows; i += kWarps * 32)
        s_unit[i] = unit_of(row0 + i, s_range[0], s_range[1] + 1);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LANES, part = lane % LANES;
    const int which = part / CPR, ch = part % CPR;
    const uint4 *src_base = which ? v : k;
    uint4 *dst_base = which ? vout : kout;
    constexpr int kStep = kWarps * ROWS_PER_PASS;
    for (int r0 = warp * ROWS_PER_PASS + sub; r0 < nrows; r0 += kStep * kUnroll) {
        uint4 buf[kUnroll];
        long long dst[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int r = r0 + q * kStep;
            ok[q] = false;
            if (r < nrows) {
                const UnitInfo U = unit_info(P, s_unit[r], P.cu);
                const long long row = row0 + r;
                int tok = -1;
                if (B.block_layers == 0) {
                    tok = sel[row];
                } else {
                    const long long ub = (long long)U.r * B.nblk + U.l / B.block_layers;
                    const long long i = row - offsets[s_unit[r]];
                    if (i < B.offsets[ub + 1] - B.offsets[ub]) tok = B.sel[B.offsets[ub] + i];
                }
                if (tok >= 0 && tok < U.n &&
                    in_range(U.kv_row0 + tok, kv_rows_total(P), nullptr)) {
                    buf[q] = ld_nc(src_base + (U.kv_row0 + tok) * CPR + ch);
                    dst[q] = row * CPR + ch;
                    ok[q] = true;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q)
            if (ok[q]) st_cs(dst_base + dst[q], buf[q]);
    }
}

// Copies output rows [r0, r1) with the kWarps warps of the calling CTA, kUnroll
// rows in flight per warp, for a caller that walks long row ranges (the fused
// kernel): no shared memory and no CTA barrier.  Each warp finds the unit of its
// first row by binary search in the offsets table, then, its rows increasing,
// advances the unit while a row lies past it (rows past the last unit are
// skipped, as are out-of-range indices).
template <int D, int kWarps, int kUnroll>
__device__ __forceinline__ void compact_rows(const DevProblem &P, const uint4 *__restrict__ k,
                                             const uint4 *__restrict__ v,
                                             const int32_t *__restrict__ sel,
                                             const int64_t *__restrict__ offsets,
                                             long long r0, long long r1,
                                             uint4 *__restrict__ kout,
                                             uint4 *__restrict__ vout) {
    constexpr int CPR = D / 8;                    // 16-byte chunks per row
    constexpr int LANES = 2 * CPR;                // K chunks then V chunks
    constexpr int ROWS_PER_PASS = 32 / LANES;     // rows one warp covers per step
    static_assert(32 % LANES == 0, "row must split evenly over a warp");
    constexpr int kStep = kWarps * ROWS_PER_PASS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LANES, part = lane % LANES;
    const int which = part / CPR, ch = part % CPR;
    const uint4 *src_base = which ? v : k;
    uint4 *dst_base = which ? vout : kout;
    const long long first = r0 + warp * ROWS_PER_PASS + sub;
    if (first >= r1) return;
    long long lo = 0, hi = P.units;              // offsets[lo] <= first < offsets[hi]
    while (hi - lo > 1) {
        const long long mid = (lo + hi) >> 1;
        if (offsets[mid] <= first) lo = mid; else hi = mid;
    }
    long long u = lo, u_end = offsets[u + 1];
    UnitInfo U = unit_info(P, u, P.cu);
    constexpr long long kIter = (long long)kStep * kUnroll;   // rows a warp step covers
    // software pipeline: the indices of the next step load while this step's rows copy
    int toks[kUnroll];
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
        const long long row = first + (long long)q * kStep;
        toks[q] = row < r1 ? sel[row] : -1;
    }
    for (long long rb = first; rb < r1; rb += kIter) {
        uint4 buf[kUnroll];
        long long dst[kUnroll];
        bool ok[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const long long row = rb + (long long)q * kStep;
            ok[q] = false;
            if (row < r1) {
                // never past the last unit, whatever total_rows the caller gave
                while (row >= u_end && u + 1 < P.units) {
                    ++u;
                    u_end = offsets[u + 1];
                    U = unit_info(P, u, P.cu);
                }
                const int tok = row < u_end ? toks[q] : -1;
                if (tok >= 0 && tok < U.n &&
                    in_range(U.kv_row0 + tok, kv_rows_total(P), nullptr)) {
                    buf[q] = ld_nc(src_base + (U.kv_row0 + tok) * CPR + ch);
                    dst[q] = row * CPR + ch;
                    ok[q] = true;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const long long row = rb + kIter + (long long)q * kStep;
            toks[q] = row < r1 ? sel[row] : -1;
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q)
            if (ok[q]) st_cs(dst_base + dst[q], buf[q]);
    }
}

}  // namespace kvevict
