// kv_compact.cu -- ragged gather of the kept K/V rows into one packed cache.
//
// Output row i of unit u (offsets[u] <= i < offsets[u+1]) is the K (and V)
// row of token sel[i] of that unit: a bit copy (GraceKV, "physical cache
// packing": one cache of its own length per layer-KV-head).  Each CTA copies a
// contiguous range of output rows, finding each row's unit by binary search in
// the offsets table between the units of its first and last rows; a warp moves one
// row pair (K and V) per step in 16-byte vectors, four rows in flight, with
// read-only loads and streaming stores (the copy is touched once).
#include "kv_internal.cuh"

namespace kvevict {
namespace {

constexpr int kRowsPerCta = 256;
constexpr int kWarps = 8;
constexpr int kUnroll = 4;

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

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
compact_kernel(DevProblem P, const uint4 *__restrict__ k, const uint4 *__restrict__ v,
               const int32_t *__restrict__ sel, const int64_t *__restrict__ offsets,
               long long total_rows, uint4 *__restrict__ kout, uint4 *__restrict__ vout) {
    constexpr int CPR = D / 8;                    // 16-byte chunks per row
    constexpr int LANES = 2 * CPR;                // K chunks then V chunks
    constexpr int ROWS_PER_PASS = 32 / LANES;     // rows one warp covers per step
    static_assert(32 % LANES == 0, "row must split evenly over a warp");
    __shared__ long long s_unit[kRowsPerCta];
    __shared__ long long s_range[2];
    const long long row0 = (long long)blockIdx.x * kRowsPerCta;
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
    for (int i = threadIdx.x; i < nrows; i += blockDim.x)
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
                const int tok = sel[row];
                if (tok >= 0 && tok < U.n) {
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

}  // namespace

cudaError_t launch_compact(const DevProblem &P, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                           const int32_t *sel, const int64_t *offsets, long long total_rows,
                           __nv_bfloat16 *kout, __nv_bfloat16 *vout, cudaStream_t s) {
    const long long blocks = (total_rows + kRowsPerCta - 1) / kRowsPerCta;
    if (blocks <= 0) return cudaSuccess;
    auto kk = reinterpret_cast<const uint4 *>(k);
    auto vv = reinterpret_cast<const uint4 *>(v);
    auto ko = reinterpret_cast<uint4 *>(kout);
    auto vo = reinterpret_cast<uint4 *>(vout);
    if (P.d == 64)
        compact_kernel<64><<<(unsigned)blocks, kWarps * 32, 0, s>>>(P, kk, vv, sel, offsets,
                                                                    total_rows, ko, vo);
    else
        compact_kernel<128><<<(unsigned)blocks, kWarps * 32, 0, s>>>(P, kk, vv, sel, offsets,
                                                                     total_rows, ko, vo);
    return cudaGetLastError();
}

}  // namespace kvevict
