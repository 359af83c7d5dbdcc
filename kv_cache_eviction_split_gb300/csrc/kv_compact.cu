// kv_compact.cu -- the stand-alone compaction kernels: the plain form
// (compact_rows over 1024-row ranges, one range per CTA) and the block-eviction
// form (compact_block, kv_compact.cuh).
#include "kv_compact.cuh"

namespace kvevict {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 4;
constexpr long long kRangeRows = 1024;   // output rows per CTA in the plain form
constexpr int kRangeUnroll = 8;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
compact_range_kernel(DevProblem P, const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                     const int32_t *__restrict__ sel, const int64_t *__restrict__ offsets,
                     long long total_rows, uint4 *__restrict__ kout, uint4 *__restrict__ vout) {
    const long long r0 = (long long)blockIdx.x * kRangeRows;
    compact_rows<D, kWarps, kRangeUnroll>(P, k, v, sel, offsets, r0,
                                          min(total_rows, r0 + kRangeRows), kout, vout);
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
compact_kernel(DevProblem P, const uint4 *__restrict__ k, const uint4 *__restrict__ v,
               const int32_t *__restrict__ sel, const int64_t *__restrict__ offsets,
               long long total_rows, uint4 *__restrict__ kout, uint4 *__restrict__ vout,
               const BlockSel B) {
    __shared__ long long s_unit[kRowsPerCta];
    __shared__ long long s_range[2];
    compact_block<D, kWarps, kUnroll>(P, k, v, sel, offsets, total_rows, kout, vout, B,
                                      blockIdx.x, s_unit, s_range);
}

cudaError_t launch_compact_any(const DevProblem &P, const __nv_bfloat16 *k,
                               const __nv_bfloat16 *v, const int32_t *sel,
                               const int64_t *offsets, long long total_rows,
                               __nv_bfloat16 *kout, __nv_bfloat16 *vout, const BlockSel &B,
                               cudaStream_t s) {
    const long long blocks = (total_rows + kRowsPerCta - 1) / kRowsPerCta;
    if (blocks <= 0) return cudaSuccess;
    auto kk = reinterpret_cast<const uint4 *>(k);
    auto vv = reinterpret_cast<const uint4 *>(v);
    auto ko = reinterpret_cast<uint4 *>(kout);
    auto vo = reinterpret_cast<uint4 *>(vout);
    if (B.block_layers == 0) {
        const long long ranges = (total_rows + kRangeRows - 1) / kRangeRows;
        if (P.d == 64)
            compact_range_kernel<64><<<(unsigned)ranges, kWarps * 32, 0, s>>>(
                P, kk, vv, sel, offsets, total_rows, ko, vo);
        else
            compact_range_kernel<128><<<(unsigned)ranges, kWarps * 32, 0, s>>>(
                P, kk, vv, sel, offsets, total_rows, ko, vo);
        return cudaGetLastError();
    }
    if (P.d == 64)
        compact_kernel<64><<<(unsigned)blocks, kWarps * 32, 0, s>>>(P, kk, vv, sel, offsets,
                                                                    total_rows, ko, vo, B);
    else
        compact_kernel<128><<<(unsigned)blocks, kWarps * 32, 0, s>>>(P, kk, vv, sel, offsets,
                                                                     total_rows, ko, vo, B);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact(const DevProblem &P, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                           const int32_t *sel, const int64_t *offsets, long long total_rows,
                           __nv_bfloat16 *kout, __nv_bfloat16 *vout, cudaStream_t s) {
    return launch_compact_any(P, k, v, sel, offsets, total_rows, kout, vout,
                              BlockSel{nullptr, nullptr, 0, 0}, s);
}

cudaError_t launch_compact_blocks(const DevProblem &P, int block_layers, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const int32_t *block_sel,
                                  const int64_t *block_offsets, const int64_t *offsets,
                                  long long total_rows, __nv_bfloat16 *kout,
                                  __nv_bfloat16 *vout, cudaStream_t s) {
    return launch_compact_any(P, k, v, nullptr, offsets, total_rows, kout, vout,
                              BlockSel{block_sel, block_offsets, block_layers,
                                       P.L / block_layers}, s);
}

}  // namespace kvevict
