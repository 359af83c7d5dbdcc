// kv_heads.cu -- per-head budgets from the scores (AdaDropKV).
//
// DropKV page, Key Contributions ("Adaptive head budgets"): DropKV scoring
// combined with AdaKV's head budget allocation.  For every (request, layer),
// every head keeps its sinks and window, and the layer's remaining slots
// k = sum_h (b_h - s - w) go to the largest middle-candidate scores of all H
// heads together, equal scores to the lower head, then the lower index; a
// head's budget is s + w + the slots it won.
//
// The layer-wide k-th largest is found by an MSB radix select over the score
// bit patterns (non-negative floats order as uint32), 8 bits a pass, run as
// short launches that are parallel over (layer, head, 16384-key chunk):
//   hb_hist_kernel  x4  histogram of the next 8 bits among the candidates that
//                       match the digits found so far, into a per-layer global
//                       histogram
//   hb_count_kernel     per head, the candidates above the threshold theta and
//                       equal to it
//   hb_final_kernel     per layer, theta's rank, the heads' budgets and offsets
// Each kernel replays the digits of the earlier passes from the stored
// histograms (one warp, identical in every CTA), so no kernel sits between the
// passes.
#include "kv_internal.cuh"

namespace kvevict {
namespace {

constexpr int kHbThreads = 512;
constexpr int kHbChunk = 16384;      // middle keys of one head per CTA
constexpr unsigned kFull = 0xffffffffu;

// k of the layer of unit u0 (its first head) from the input budgets; false if a
// budget is outside [s + w, n] or disagrees with the offsets.
__device__ bool layer_k(const DevProblem &P, long long u0, int n, const int32_t *budgets,
                        const int64_t *offsets, long long &k) {
    k = 0;
    bool ok = true;
    for (int h = 0; h < P.H; ++h) {
        const long long b = budgets[u0 + h];
        ok = ok && b >= (long long)P.sinks + P.w && b <= n &&
             offsets[u0 + h + 1] - offsets[u0 + h] == b;
        k += b - P.sinks - P.w;
    }
    return ok;
}

// The digits of passes 0 .. passes-1, replayed by one full warp from the layer's
// histograms hist[pass][256]: prefix and mask of the matched bits, and the rank
// still to find among the candidates that match them.
__device__ void replay(const unsigned *hist, int passes, unsigned &prefix, unsigned &mask,
                       unsigned &remaining) {
    const int lane = threadIdx.x & 31;
    for (int p = 0; p < passes; ++p) {
        const unsigned *hp = hist + p * 256;
        // lane l holds bins 255 - 8l down to 248 - 8l (descending digits)
        unsigned c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = hp[255 - 8 * lane - i];
            sum += c[i];
        }
        unsigned incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned y = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += y;
        }
        const unsigned excl = incl - sum;
        const bool mine = excl < remaining && remaining <= incl;
        const unsigned who = __ballot_sync(kFull, mine);
        unsigned digit = 0, above = 0;
        if (mine) {
            unsigned acc = excl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (acc + c[i] >= remaining) {
                    digit = 255u - 8u * lane - i;
                    above = acc;
                    break;
                }
                acc += c[i];
            }
        }
        const int src = who ? __ffs(who) - 1 : 0;
        digit = who ? __shfl_sync(kFull, digit, src) : 0u;
        above = who ? __shfl_sync(kFull, above, src) : 0u;
        const int shift = 24 - 8 * p;
        remaining -= above;
        prefix |= digit << shift;
        mask |= 255u << shift;
    }
}

struct HbCta {
    long long u;        // unit (request, layer, head) of the CTA
    long long rl;       // request * L + layer
    int j0, j1;         // middle keys [j0, j1) of the CTA
};

__device__ __forceinline__ HbCta hb_cta(const DevProblem &P, int cph) {
    HbCta c;
    const int chunk = (int)(blockIdx.x % cph);
    c.u = blockIdx.x / cph;
    c.rl = c.u / P.H;
    const UnitInfo U = unit_info(P, c.u, P.cu);
    c.j0 = P.sinks + chunk * kHbChunk;
    c.j1 = min(U.n - P.w, c.j0 + kHbChunk);
    return c;
}

// Warp 0: whether the layer needs the select (valid budgets, 0 < k < candidates)
// and, if so, the digits of the first `passes` passes; shared with the CTA.
__device__ bool hb_setup(const DevProblem &P, const HbCta &c, const int32_t *budgets,
                         const int64_t *offsets, const unsigned *hist, int passes,
                         unsigned *s_prefix, unsigned *s_mask, int *s_run) {
    if (threadIdx.x < 32) {
        const long long u0 = c.rl * P.H;
        const int n = (int)(P.cu[c.rl / P.L + 1] - P.cu[c.rl / P.L]);
        long long k;
        const bool ok = layer_k(P, u0, n, budgets, offsets, k);
        const long long cand = (long long)(n - P.w - P.sinks) * P.H;
        const bool run = ok && k > 0 && k < cand;
        unsigned prefix = 0, mask = 0, remaining = (unsigned)(run ? k : 0);
        if (run) replay(hist + c.rl * 1024, passes, prefix, mask, remaining);
        if (threadIdx.x == 0) {
            *s_run = run;
            *s_prefix = prefix;
            *s_mask = mask;
        }
    }
    __syncthreads();
    return *s_run != 0;
}

__global__ void __launch_bounds__(kHbThreads)
hb_hist_kernel(const DevProblem P, const float *__restrict__ scores,
               const int32_t *__restrict__ budgets, const int64_t *__restrict__ offsets,
               unsigned *__restrict__ hist_g, int pass, int cph) {
    __shared__ unsigned hist[256];
    __shared__ unsigned s_prefix, s_mask;
    __shared__ int s_run;
    const HbCta c = hb_cta(P, cph);
    if (c.j0 >= c.j1) return;
    for (int i = threadIdx.x; i < 256; i += kHbThreads) hist[i] = 0;
    if (!hb_setup(P, c, budgets, offsets, hist_g, pass, &s_prefix, &s_mask, &s_run)) return;
    const unsigned prefix = s_prefix, mask = s_mask;
    const int shift = 24 - 8 * pass;
    const UnitInfo U = unit_info(P, c.u, P.cu);
    const unsigned *keys = reinterpret_cast<const unsigned *>(scores + U.kv_row0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // each warp takes 4 x 32 consecutive keys a step, all four loads in flight first
    for (int jb = c.j0 + 128 * warp; jb < c.j1; jb += 4 * kHbThreads) {
        unsigned key[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = jb + 32 * q + lane;
            key[q] = j < c.j1 ? __ldg(keys + j) : 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (jb + 32 * q + lane < c.j1 && (key[q] & mask) == prefix)
                atomicAdd(&hist[(key[q] >> shift) & 255u], 1u);
    }
    __syncthreads();
    unsigned *out = hist_g + c.rl * 1024 + pass * 256;
    for (int i = threadIdx.x; i < 256; i += kHbThreads)
        if (hist[i]) atomicAdd(out + i, hist[i]);
}

__global__ void __launch_bounds__(kHbThreads)
hb_count_kernel(const DevProblem P, const float *__restrict__ scores,
                const int32_t *__restrict__ budgets, const int64_t *__restrict__ offsets,
                const unsigned *__restrict__ hist_g, unsigned *__restrict__ cnt, int cph) {
    __shared__ unsigned s_prefix, s_mask;
    __shared__ int s_run;
    __shared__ unsigned red[2][kHbThreads / 32];
    const HbCta c = hb_cta(P, cph);
    if (c.j0 >= c.j1) return;
    if (!hb_setup(P, c, budgets, offsets, hist_g, 4, &s_prefix, &s_mask, &s_run)) return;
    const unsigned theta = s_prefix;
    const UnitInfo U = unit_info(P, c.u, P.cu);
    const unsigned *keys = reinterpret_cast<const unsigned *>(scores + U.kv_row0);
    unsigned above = 0, eq = 0;
    for (int jb = c.j0 + threadIdx.x; jb < c.j1; jb += 4 * kHbThreads) {
        unsigned key[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = jb + q * kHbThreads;
            key[q] = j < c.j1 ? __ldg(keys + j) : 0u;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = jb + q * kHbThreads < c.j1;
            above += in && key[q] > theta;
            eq += in && key[q] == theta;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        above += __shfl_xor_sync(kFull, above, off);
        eq += __shfl_xor_sync(kFull, eq, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        red[0][warp] = above;
        red[1][warp] = eq;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned a = 0, e = 0;
        for (int i = 0; i < kHbThreads / 32; ++i) {
            a += red[0][i];
            e += red[1][i];
        }
        if (a) atomicAdd(cnt + 2 * c.u, a);
        if (e) atomicAdd(cnt + 2 * c.u + 1, e);
    }
}

// One warp per layer: the heads' budgets and offsets.
__global__ void __launch_bounds__(32)
hb_final_kernel(const DevProblem P, const int32_t *__restrict__ budgets,
                const int64_t *__restrict__ offsets, const unsigned *__restrict__ hist_g,
                const unsigned *__restrict__ cnt, int32_t *__restrict__ budgets_out,
                int64_t *__restrict__ offsets_out, int *status) {
    const long long rl = blockIdx.x;
    const long long u0 = rl * P.H;
    const int lane = threadIdx.x;
    const int n = (int)(P.cu[rl / P.L + 1] - P.cu[rl / P.L]);
    long long k;
    const bool ok = layer_k(P, u0, n, budgets, offsets, k);
    const bool last = u0 + P.H == P.units;
    if (!ok) {
        for (int h = lane; h < P.H; h += 32) {
            budgets_out[u0 + h] = budgets[u0 + h];
            offsets_out[u0 + h] = offsets[u0 + h];
        }
        if (lane == 0) {
            post_status(status, KV_ERR_BUDGET);
            if (last) offsets_out[P.units] = offsets[P.units];
        }
        return;
    }
    const int m = n - P.w - P.sinks;             // middle candidates per head
    const long long cand = (long long)m * P.H;
    unsigned prefix = 0, mask = 0, remaining = (unsigned)(k > 0 && k < cand ? k : 0);
    if (k > 0 && k < cand) replay(hist_g + rl * 1024, 4, prefix, mask, remaining);
    if (lane == 0) {
        long long eq_left = remaining;           // ties at theta, to the lower heads first
        long long running = offsets[u0];
        const int keep = P.sinks + P.w;
        for (int h = 0; h < P.H; ++h) {
            long long c;
            if (k <= 0) {
                c = 0;
            } else if (k >= cand) {
                c = m;
            } else {
                const long long eq = cnt[2 * (u0 + h) + 1];
                const long long take = eq_left < eq ? eq_left : eq;
                eq_left -= take;
                c = (long long)cnt[2 * (u0 + h)] + take;
            }
            budgets_out[u0 + h] = (int32_t)(keep + c);
            offsets_out[u0 + h] = running;
            running += keep + c;
        }
        if (last) offsets_out[P.units] = running;
    }
}

}  // namespace

size_t head_budget_ws_bytes(const DevProblem &P) {
    const size_t rl = (size_t)(P.units / (P.H > 0 ? P.H : 1));
    return rl * 1024 * sizeof(unsigned) + (size_t)P.units * 2 * sizeof(unsigned);
}

cudaError_t launch_head_budgets(const DevProblem &P, const float *scores, const int32_t *budgets,
                                const int64_t *offsets, int32_t *budgets_out,
                                int64_t *offsets_out, int *status, void *scratch,
                                cudaStream_t s) {
    const long long rl = P.units / P.H;
    unsigned *hist = static_cast<unsigned *>(scratch);
    unsigned *cnt = hist + rl * 1024;
    cudaError_t e = cudaMemsetAsync(scratch, 0, head_budget_ws_bytes(P), s);
    if (e != cudaSuccess) return e;
    const int mid_max = P.max_n - P.w - P.sinks;
    const int cph = mid_max > 0 ? (mid_max + kHbChunk - 1) / kHbChunk : 1;
    const long long grid = P.units * cph;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    for (int pass = 0; pass < 4; ++pass)
        hb_hist_kernel<<<(unsigned)grid, kHbThreads, 0, s>>>(P, scores, budgets, offsets, hist,
                                                             pass, cph);
    hb_count_kernel<<<(unsigned)grid, kHbThreads, 0, s>>>(P, scores, budgets, offsets, hist, cnt,
                                                          cph);
    hb_final_kernel<<<(unsigned)rl, 32, 0, s>>>(P, budgets, offsets, hist, cnt, budgets_out,
                                                offsets_out, status);
    return cudaGetLastError();
}

}  // namespace kvevict
