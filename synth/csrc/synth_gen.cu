// synth_gen.cu -- device twin of the host generator in synth/__init__.py.
//
// Fills the packed K and V tensors ([L][H][N_tot][d], bf16) of a synthetic
// workload with the same bits the numpy generator produces: element e of a
// stream with key `key` takes the words mix64(key + (3e + i + 1) * PHI),
// i = 0, 1, 2 (splitmix64's output function), sums their twelve 16-bit
// fields (Irwin-Hall(12)), centres and scales by 2^-16 exactly, multiplies by
// a power-of-two scale and rounds to bf16 (nearest, ties to even).  Then
// overwrites the heavy key rows with rows computed on the host.
//
// Input generation only: nothing of the eviction method lives here.
#include <cstdint>

#include <cuda_runtime.h>

namespace {

constexpr unsigned long long kPhi = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ unsigned short normal_bf16(unsigned long long key, unsigned long long e,
                                                      float scale) {
    long long acc = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const unsigned long long w = mix64(key + (3ull * e + (unsigned long long)i + 1ull) * kPhi);
        acc += (long long)(w & 0xFFFFull) + (long long)((w >> 16) & 0xFFFFull) +
               (long long)((w >> 32) & 0xFFFFull) + (long long)(w >> 48);
    }
    const float z = __int2float_rn((int)(acc - 393210)) * (1.0f / 65536.0f);
    unsigned int b = __float_as_uint(__fmul_rn(z, scale));
    b = b + 0x7FFFu + ((b >> 16) & 1u);
    return (unsigned short)(b >> 16);
}

__global__ void fill_kv_kernel(uint4 *__restrict__ k, uint4 *__restrict__ v, int H,
                               long long N_tot, int d, unsigned long long key_k,
                               unsigned long long key_v, float sigma,
                               const int *__restrict__ outliers, int n_out, float out_scale,
                               long long n_vec) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n_vec; t += stride) {
        const unsigned long long e0 = (unsigned long long)t * 8ull;
        const long long row = (long long)(e0 / (unsigned long long)d);
        const int c0 = (int)(e0 % (unsigned long long)d);
        const long long lh = row / N_tot;
        const int *oc = outliers + lh * n_out;
        unsigned short hk[8], hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float sc = sigma;
            for (int j = 0; j < n_out; ++j)
                if (oc[j] == c0 + i) sc = sigma * out_scale;
            hk[i] = normal_bf16(key_k, e0 + i, sc);
            hv[i] = normal_bf16(key_v, e0 + i, sc);
        }
        uint4 pk, pv;
        pk.x = hk[0] | ((unsigned)hk[1] << 16); pk.y = hk[2] | ((unsigned)hk[3] << 16);
        pk.z = hk[4] | ((unsigned)hk[5] << 16); pk.w = hk[6] | ((unsigned)hk[7] << 16);
        pv.x = hv[0] | ((unsigned)hv[1] << 16); pv.y = hv[2] | ((unsigned)hv[3] << 16);
        pv.z = hv[4] | ((unsigned)hv[5] << 16); pv.w = hv[6] | ((unsigned)hv[7] << 16);
        k[t] = pk;
        v[t] = pv;
    }
}

__global__ void place_heavy_kernel(unsigned short *__restrict__ k, int L, int H, long long N_tot,
                                   int d, const long long *__restrict__ cu,
                                   const int *__restrict__ pos, int nh,
                                   const unsigned short *__restrict__ rows) {
    const long long item = blockIdx.x;          // ((r * L + l) * H + h) * nh + i
    const long long seg = item / nh;
    const int h = (int)(seg % H);
    const int l = (int)((seg / H) % L);
    const int r = (int)(seg / ((long long)H * L));
    const long long tok = cu[r] + pos[item];
    unsigned short *dst = k + (((long long)l * H + h) * N_tot + tok) * d;
    const unsigned short *src = rows + seg * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) dst[c] = src[c];
}

}  // namespace

extern "C" {

// Returns 0 or a cudaError_t code.  k, v: bf16 [L][H][N_tot][d] (16-byte aligned,
// d a multiple of 8); outliers: device int32 [L][H][n_out].
int synth_fill_kv(void *k, void *v, int L, int H, long long N_tot, int d,
                  unsigned long long key_k, unsigned long long key_v, float sigma,
                  const int *outliers, int n_out, float out_scale, void *stream) {
    const long long n_vec = (long long)L * H * N_tot * d / 8;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n_vec + 255) / 256;
    if (blocks > (long long)sms * 32) blocks = (long long)sms * 32;
    if (blocks < 1) blocks = 1;
    fill_kv_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
        (uint4 *)k, (uint4 *)v, H, N_tot, d, key_k, key_v, sigma, outliers, n_out, out_scale,
        n_vec);
    return (int)cudaGetLastError();
}

// Overwrites K rows: for each (r, l, h, i), row cu[r] + pos[r][l][h][i] of
// (l, h) receives rows[r][l][h][:].  All pointers are device memory.
int synth_place_heavy(void *k, int R, int L, int H, long long N_tot, int d, const long long *cu,
                      const int *pos, int nh, const void *rows, void *stream) {
    const long long items = (long long)R * L * H * nh;
    if (items == 0) return 0;
    place_heavy_kernel<<<(unsigned)items, 128, 0, (cudaStream_t)stream>>>(
        (unsigned short *)k, L, H, N_tot, d, cu, pos, nh, (const unsigned short *)rows);
    return (int)cudaGetLastError();
}

}  // extern "C"
