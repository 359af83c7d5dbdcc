// kv_compact.cu -- ragged gather of the kept K/V rows into one packed cache.
//
// Output row i of unit u (offsets[u] <= i < offsets[u+1]) is the K (and V)
// row of token sel[i] of that unit: a bit copy in 16-byte vectors.  Work items
// are 16-byte chunks ordered row-major over (row, K|V, chunk), so the threads
// of a warp copy consecutive bytes of one or two rows; each finds its unit by
// binary search in the offsets table.
#include "kv_internal.cuh"

namespace kvevict {
namespace {

template <int D>
__global__ void __launch_bounds__(256)
compact_kernel(DevProblem P, const uint4 *__restrict__ k, const uint4 *__restrict__ v,
               const int32_t *__restrict__ sel, const int64_t *__restrict__ offsets,
               long long total_rows, uint4 *__restrict__ kout, uint4 *__restrict__ vout) {
    constexpr int CPR = D / 8;          // 16-byte chunks per row
    constexpr int PER_ROW = 2 * CPR;    // K chunks then V chunks
    const long long items = total_rows * PER_ROW;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += stride) {
        const long long row = it / PER_ROW;
        const int rem = (int)(it % PER_ROW);
        const int which = rem / CPR, ch = rem % CPR;
        long long lo = 0, hi = P.units;   // offsets[lo] <= row < offsets[hi]
        while (hi - lo > 1) {
            const long long mid = (lo + hi) >> 1;
            if (offsets[mid] <= row) lo = mid; else hi = mid;
        }
        const UnitInfo U = unit_info(P, lo, P.cu);
        const int tok = sel[row];
        if (tok < 0 || tok >= U.n) continue;
        const long long src = (U.kv_row0 + tok) * CPR + ch;
        const long long dst = row * CPR + ch;
        if (which) vout[dst] = __ldg(v + src);
        else kout[dst] = __ldg(k + src);
    }
}

}  // namespace

cudaError_t launch_compact(const DevProblem &P, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                           const int32_t *sel, const int64_t *offsets, long long total_rows,
                           __nv_bfloat16 *kout, __nv_bfloat16 *vout, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long items = total_rows * 2 * (P.d / 8);
    long long blocks = (items + 255) / 256;
    blocks = blocks < (long long)sms * 16 ? blocks : (long long)sms * 16;
    if (blocks < 1) blocks = 1;
    auto kk = reinterpret_cast<const uint4 *>(k);
    auto vv = reinterpret_cast<const uint4 *>(v);
    auto ko = reinterpret_cast<uint4 *>(kout);
    auto vo = reinterpret_cast<uint4 *>(vout);
    if (P.d == 64)
        compact_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(P, kk, vv, sel, offsets, total_rows, ko, vo);
    else
        compact_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(P, kk, vv, sel, offsets, total_rows, ko, vo);
    return cudaGetLastError();
}

}  // namespace kvevict
