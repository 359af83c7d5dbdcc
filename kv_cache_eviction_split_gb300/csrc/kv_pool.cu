// kv_pool.cu -- 1-D max pooling of the scores before selection.
//
// DropKV, "Methodology in Plain English": the scores are max-pooled over
// neighbouring tokens after the SnapKV convention (kernel 11 in its
// evaluation); the BellowsKV blog takes the maximum over a 13-position window
// centred on each token.  Pooling runs per unit over the keys outside the
// observation window, [0, n - w); the w window keys are kept by selection
// anyway and are copied unchanged.
//
// HBM-bound: one read and one write of every score.  A CTA takes a tile of
// 4096 packed tokens of one (layer, KV head) score row plus a halo of r on
// each side into shared memory with coalesced loads (16 per thread in flight);
// each thread pools 16 consecutive tokens from registers (one request and all candidates: no
// masks), or, near a request end or the window, with per-token bounds; the
// results go back through shared memory so the stores are coalesced too.
#include <cfloat>

#include "kv_internal.cuh"

namespace kvevict {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kPoolPer = 16;
constexpr int kPoolTile = kPoolThreads * kPoolPer;   // tokens per CTA
constexpr int kMaxRadius = 127;                      // kernel <= 255
constexpr int kXs = kPoolTile + 2 * kMaxRadius + 8;  // halo + float4 over-read

// Index of the request holding packed token t: cu[r] <= t < cu[r + 1].
__device__ __forceinline__ int find_request(const long long *cu, int R, long long t) {
    int lo = 0, hi = R;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// RAD >= 0: radius known at compile time, windows read into registers;
// RAD < 0: radius `rad_rt`, windows read from shared memory.
template <int RAD>
__global__ void __launch_bounds__(kPoolThreads, 4)
pool_kernel(const DevProblem P, int rad_rt, const float *__restrict__ in, float *__restrict__ out,
            long long tiles_per_row) {
    __shared__ __align__(16) float xs[kXs];
    __shared__ __align__(16) float ys[kPoolTile];
    const int rad = RAD >= 0 ? RAD : rad_rt;
    const long long row = blockIdx.x / tiles_per_row;          // l * H + h
    const long long t0 = (blockIdx.x % tiles_per_row) * kPoolTile;
    const long long N = P.N_tot;
    const float *rin = in + row * N;
    float *rout = out + row * N;
    const int tid = threadIdx.x;

    // xs[s] = score of packed token t0 - rad + s (-inf outside the row): every load
    // of the thread is issued before the first shared-memory store
    constexpr int kLoads = (kXs + kPoolThreads - 1) / kPoolThreads;
    float ld[kLoads];
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
        const int s = tid + q * kPoolThreads;
        const long long t = t0 - rad + s;
        ld[q] = (s < kPoolTile + 2 * rad && t >= 0 && t < N) ? __ldg(rin + t) : -INFINITY;
    }
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
        const int s = tid + q * kPoolThreads;
        if (s < kXs) xs[s] = ld[q];
    }
    __syncthreads();

    const long long j0 = t0 + (long long)kPoolPer * tid;   // first token of this thread
    float y[kPoolPer];
    if (j0 < N) {
        int r = find_request(P.cu, P.R, j0);
        long long lo = P.cu[r], hi = P.cu[r + 1] - P.w;       // candidates [lo, hi)
        const float *xw = xs + kPoolPer * tid;                  // xw[k]: token j0 - rad + k
        const bool fast = j0 - rad >= lo && j0 + kPoolPer - 1 + rad < hi;
        if constexpr (RAD >= 0) {
            constexpr int W = kPoolPer + 2 * RAD;
            float x[(W + 3) / 4 * 4];
#pragma unroll
            for (int q = 0; q < (W + 3) / 4; ++q) {
                const float4 v = reinterpret_cast<const float4 *>(xw)[q];
                x[4 * q] = v.x;
                x[4 * q + 1] = v.y;
                x[4 * q + 2] = v.z;
                x[4 * q + 3] = v.w;
            }
            if (fast) {
#pragma unroll
                for (int e = 0; e < kPoolPer; ++e) {
                    float m = x[e];
#pragma unroll
                    for (int k = 1; k <= 2 * RAD; ++k) m = fmaxf(m, x[e + k]);
                    y[e] = m;
                }
            } else {
#pragma unroll
                for (int e = 0; e < kPoolPer; ++e) {
                    const long long j = j0 + e;
                    while (r + 1 < P.R && j >= P.cu[r + 1]) {
                        ++r;
                        lo = P.cu[r];
                        hi = P.cu[r + 1] - P.w;
                    }
                    float m = x[e + RAD];
                    if (j < hi) {
#pragma unroll
                        for (int k = -RAD; k <= RAD; ++k)
                            if (j + k >= lo && j + k < hi) m = fmaxf(m, x[e + RAD + k]);
                    }
                    y[e] = m;
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < kPoolPer; ++e) {
                const long long j = j0 + e;
                if (!fast) {
                    while (r + 1 < P.R && j >= P.cu[r + 1]) {
                        ++r;
                        lo = P.cu[r];
                        hi = P.cu[r + 1] - P.w;
                    }
                }
                float m = xw[e + rad];
                if (fast) {
                    for (int k = 0; k <= 2 * rad; ++k) m = fmaxf(m, xw[e + k]);
                } else if (j < hi) {
                    for (int k = -rad; k <= rad; ++k)
                        if (j + k >= lo && j + k < hi) m = fmaxf(m, xw[e + rad + k]);
                }
                y[e] = m;
            }
        }
        float4 *yv = reinterpret_cast<float4 *>(ys + kPoolPer * tid);
#pragma unroll
        for (int q = 0; q < kPoolPer / 4; ++q)
            yv[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
    }
    __syncthreads();
    for (int s = tid; s < kPoolTile; s += kPoolThreads) {
        const long long t = t0 + s;
        if (t < N) rout[t] = ys[s];
    }
}

template <int RAD>
void launch_pool_rad(const DevProblem &P, int rad, const float *in, float *out,
                     cudaStream_t st) {
    const long long tiles = (P.N_tot + kPoolTile - 1) / kPoolTile;
    const long long blocks = tiles * P.L * P.H;
    pool_kernel<RAD><<<(unsigned)blocks, kPoolThreads, 0, st>>>(P, rad, in, out, tiles);
}

}  // namespace

cudaError_t launch_pool(const DevProblem &P, int kernel, const float *in, float *out,
                        cudaStream_t s) {
    if (P.N_tot == 0) return cudaSuccess;
    const long long tiles = (P.N_tot + kPoolTile - 1) / kPoolTile;
    if (tiles * P.L * P.H > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int rad = (kernel - 1) / 2;
    switch (rad) {
        case 0: launch_pool_rad<0>(P, rad, in, out, s); break;
        case 1: launch_pool_rad<1>(P, rad, in, out, s); break;
        case 2: launch_pool_rad<2>(P, rad, in, out, s); break;
        case 3: launch_pool_rad<3>(P, rad, in, out, s); break;
        case 4: launch_pool_rad<4>(P, rad, in, out, s); break;
        case 5: launch_pool_rad<5>(P, rad, in, out, s); break;
        case 6: launch_pool_rad<6>(P, rad, in, out, s); break;
        case 7: launch_pool_rad<7>(P, rad, in, out, s); break;
        case 8: launch_pool_rad<8>(P, rad, in, out, s); break;
        default: launch_pool_rad<-1>(P, rad, in, out, s); break;
    }
    return cudaGetLastError();
}

}  // namespace kvevict
