// kv_blocks.cu -- block scores for block eviction (BellowsKV).
//
// BellowsKV blog, eviction operator: the eviction decision is made once per
// block of consecutive layers, from the window queries' attention weights
// summed over all layers and heads of the block.  block[b][t] = sum over the
// block's layers l (in order) and heads h (in order) of scores[l][h][t], for
// every packed token t.  HBM-bound: the scores are read once, the block scores
// written once; consecutive threads take consecutive tokens.
#include "kv_internal.cuh"

namespace kvevict {
namespace {

__global__ void __launch_bounds__(256)
block_sum_kernel(const DevProblem P, int block_layers, const float *__restrict__ scores,
                 float *__restrict__ out) {
    const long long N = P.N_tot;
    const int nblk = P.L / block_layers;
    const long long total = (long long)nblk * N;
    const long long step = (long long)gridDim.x * blockDim.x;
    const long long plane = (long long)P.H * N;          // one layer of scores
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += step) {
        const long long b = i / N, t = i - b * N;
        const float *src = scores + b * block_layers * plane + t;
        float acc = 0.f;
        for (int l = 0; l < block_layers; ++l)
            for (int h = 0; h < P.H; ++h) acc += __ldg(src + l * plane + (long long)h * N);
        out[i] = acc;
    }
}

}  // namespace

cudaError_t launch_block_sum(const DevProblem &P, int block_layers, const float *scores,
                             float *out, cudaStream_t s) {
    const long long total = (long long)(P.L / block_layers) * P.N_tot;
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (total + 255) / 256;
    const long long grid = want < (long long)sms * 16 ? want : (long long)sms * 16;
    block_sum_kernel<<<(unsigned)grid, 256, 0, s>>>(P, block_layers, scores, out);
    return cudaGetLastError();
}

}  // namespace kvevict
