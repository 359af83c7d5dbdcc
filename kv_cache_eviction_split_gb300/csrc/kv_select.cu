// kv_select.cu -- budgeted per-unit top-k with sinks and window pinned.
//
// One block per unit.  Scores are non-negative floats, so their IEEE bit
// patterns, read as uint32, order like the values.  A 4-pass MSB radix select
// (8 bits a pass) finds the exact bit pattern theta of the k-th largest
// middle candidate and how many candidates equal to theta must be taken;
// a final ordered pass keeps every candidate above theta and the first
// `need` candidates equal to theta in index order (the lower index wins a
// tie), writing the kept indices ascending between the sinks and the window.
#include "kv_internal.cuh"

namespace kvevict {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelItems = 8;
constexpr int kSelChunk = kSelThreads * kSelItems;

// Exclusive block-wide prefix sum over kSelThreads values; *total = sum.
__device__ __forceinline__ unsigned block_exclusive_scan(unsigned x, unsigned *warp_sums,
                                                         unsigned *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned t = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        warp_sums[lane] = t;
    }
    __syncthreads();
    const unsigned before = warp > 0 ? warp_sums[warp - 1] : 0u;
    *total = warp_sums[31];
    __syncthreads();
    return before + incl - x;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(DevProblem P, const float *__restrict__ scores, const int32_t *__restrict__ budgets,
              const int64_t *__restrict__ offsets, int32_t *__restrict__ sel, int *status) {
    __shared__ unsigned hist[256];
    __shared__ unsigned warp_sums[32];
    __shared__ unsigned s_digit, s_above;
    __shared__ unsigned chunk_keys[kSelChunk];

    const long long u = blockIdx.x;
    const int tid = threadIdx.x;
    const UnitInfo U = unit_info(P, u, P.cu);
    const int n = U.n;
    const long long b = budgets[u];
    const long long off = offsets[u];
    if (b < (long long)P.sinks + P.w || b > n || offsets[u + 1] - off != b) {
        if (tid == 0) post_status(status, KV_ERR_BUDGET);
        return;
    }
    int32_t *out = sel + off;
    for (int j = tid; j < P.sinks; j += kSelThreads) out[j] = j;
    for (int t = tid; t < P.w; t += kSelThreads) out[b - P.w + t] = n - P.w + t;

    const int lo = P.sinks, hi = n - P.w;
    const unsigned k = (unsigned)(b - P.sinks - P.w);
    if (k == 0) return;
    const unsigned *keys = reinterpret_cast<const unsigned *>(scores + U.kv_row0);
    if (k == (unsigned)(hi - lo)) {
        for (int j = lo + tid; j < hi; j += kSelThreads) out[P.sinks + j - lo] = j;
        return;
    }

    // ---- radix select of theta, the bit pattern of the k-th largest candidate
    unsigned prefix = 0, mask = 0, remaining = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int j = lo + tid; j < hi; j += kSelThreads) {
            const unsigned key = __ldg(keys + j);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        // reverse-order inclusive scan: incl(t) = number of candidates with digit >= 255 - t
        const unsigned h = tid < 256 ? hist[255 - tid] : 0u;
        unsigned tot;
        const unsigned excl = block_exclusive_scan(h, warp_sums, &tot);
        const unsigned incl = excl + h;
        if (tid < 256 && incl >= remaining && excl < remaining) {
            s_digit = 255u - tid;
            s_above = excl;
        }
        __syncthreads();
        remaining -= s_above;
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    const unsigned theta = prefix, need_eq = remaining;

    // ---- ordered output of the kept middle candidates
    unsigned base_sel = 0, eq_seen = 0;
    for (int c0 = lo; c0 < hi; c0 += kSelChunk) {
        const int len = min(kSelChunk, hi - c0);
        __syncthreads();
        for (int i = tid; i < len; i += kSelThreads) chunk_keys[i] = __ldg(keys + c0 + i);
        __syncthreads();
        unsigned n_eq = 0;
#pragma unroll
        for (int it = 0; it < kSelItems; ++it) {
            const int i = tid * kSelItems + it;
            if (i < len && chunk_keys[i] == theta) ++n_eq;
        }
        unsigned eq_total;
        const unsigned eq_before = block_exclusive_scan(n_eq, warp_sums, &eq_total);
        unsigned keep_bits = 0, n_keep = 0, eq_rank = eq_seen + eq_before;
#pragma unroll
        for (int it = 0; it < kSelItems; ++it) {
            const int i = tid * kSelItems + it;
            if (i >= len) break;
            const unsigned key = chunk_keys[i];
            bool keep = key > theta;
            if (key == theta) {
                keep = eq_rank < need_eq;
                ++eq_rank;
            }
            if (keep) {
                keep_bits |= 1u << it;
                ++n_keep;
            }
        }
        unsigned keep_total;
        unsigned dst = base_sel + block_exclusive_scan(n_keep, warp_sums, &keep_total);
#pragma unroll
        for (int it = 0; it < kSelItems; ++it) {
            if (keep_bits & (1u << it)) out[P.sinks + dst++] = c0 + tid * kSelItems + it;
        }
        base_sel += keep_total;
        eq_seen += eq_total;
    }
}

}  // namespace

cudaError_t launch_select(const DevProblem &P, const float *scores, const int32_t *budgets,
                          const int64_t *offsets, int32_t *sel, int *status, cudaStream_t s) {
    select_kernel<<<(unsigned)P.units, kSelThreads, 0, s>>>(P, scores, budgets, offsets, sel,
                                                            status);
    return cudaGetLastError();
}

}  // namespace kvevict
