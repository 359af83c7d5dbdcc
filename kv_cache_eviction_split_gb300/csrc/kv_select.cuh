// kv_select.cuh -- budgeted top-k of one unit, with sinks and window pinned, as
// a device function (select_unit) that the stand-alone select kernel
// (kv_select.cu, one 1024-thread CTA per unit) and the fused kernel
// (kv_fused.cu, units round-robin over persistent CTAs) call.
//
// Scores are non-negative floats, so their IEEE bit patterns, read as uint32,
// order like the values.  A 4-pass MSB radix select (8 bits a pass) finds the
// exact bit pattern theta of the k-th largest middle candidate and how many
// candidates equal to theta must be taken; a final ordered pass keeps every
// candidate above theta and the first `need` candidates equal to theta in index
// order (the lower index wins a tie), writing the kept indices ascending
// between the sinks and the window.
#pragma once
#include "kv_internal.cuh"

namespace kvevict {

constexpr int kSelItems = 8;      // candidates a thread holds in the ordered pass
constexpr int kSelLoads = 4;      // loads a thread has in flight in a radix pass (default)

// Shared memory of select_unit (kT threads).
struct SelSmem {
    unsigned *hist;         // [256]
    unsigned *warp_sums;    // [32]
    unsigned *scalars;      // [2]: digit, count above it
    unsigned *chunk_keys;   // [kT * kItems]
};

template <int kT, int kItems = kSelItems>
__host__ __device__ constexpr int sel_smem_bytes() {
    return (256 + 32 + 2 + 2 + kT * kItems) * 4;
}

// Carves SelSmem out of `base` (sel_smem_bytes<kT, kItems>() bytes, 4-byte aligned).
template <int kT>
__device__ __forceinline__ SelSmem sel_smem(void *base) {
    unsigned *b = static_cast<unsigned *>(base);
    return SelSmem{b, b + 256, b + 288, b + 292};
}

// Exclusive prefix sum over the kT threads of the block; *total = the sum.
template <int kT>
__device__ __forceinline__ unsigned sel_block_scan(unsigned x, unsigned *warp_sums,
                                                   unsigned *total) {
    constexpr int kWarps = kT / 32;
    static_assert(kT % 32 == 0 && kWarps <= 32, "block of whole warps, at most 32");
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
        unsigned t = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        warp_sums[lane] = t;
    }
    __syncthreads();
    const unsigned before = warp > 0 ? warp_sums[warp - 1] : 0u;
    *total = warp_sums[kWarps - 1];
    __syncthreads();
    return before + incl - x;
}

// A score's bit pattern: read-only (non-coherent) load, or a plain one when the
// scores were written earlier in the same kernel.
template <bool kCoherent>
__device__ __forceinline__ unsigned sel_key(const unsigned *p) {
    if constexpr (kCoherent) return *p;
    else return __ldg(p);
}

// Selection of unit u by the kT threads of the calling CTA (all call it; the
// returns are uniform), kLoads keys in flight per thread in the radix passes and
// kItems candidates per thread in each round of the ordered pass.  Budget errors
// post KV_ERR_BUDGET and write nothing.
template <int kT, bool kCoherent, int kLoads = kSelLoads, int kItems = kSelItems>
__device__ __forceinline__ void select_unit(const DevProblem &P, const float *scores,
                                            const int32_t *budgets, const int64_t *offsets,
                                            int32_t *sel, int *status, long long u,
                                            const SelSmem &sm) {
    static_assert(kT >= 256, "the digit scan needs a thread per bin");
    static_assert(kItems <= 32, "keep flags are one 32-bit word per thread");
    constexpr int kChunk = kT * kItems;
    const int tid = threadIdx.x;
    const UnitInfo U = unit_info(P, u, P.cu);
    const int n = U.n;
    const long long b = budgets[u];
    const long long off = offsets[u];
    if (b < (long long)P.sinks + P.w || b > n || offsets[u + 1] - off != b) {
        if (tid == 0) post_status(status, KV_ERR_BUDGET);
        return;
    }
    // the unit's output range and its scores lie inside their arrays
    if (!in_range(off, offsets[P.units], status) || !in_range(off + b - 1, offsets[P.units], status) ||
        !in_range(U.kv_row0 + n - 1, kv_rows_total(P), status))
        return;
    int32_t *out = sel + off;
    for (int j = tid; j < P.sinks; j += kT) out[j] = j;
    for (int t = tid; t < P.w; t += kT) out[b - P.w + t] = n - P.w + t;

    const int lo = P.sinks, hi = n - P.w;
    const unsigned k = (unsigned)(b - P.sinks - P.w);
    if (k == 0) return;
    const unsigned *keys = reinterpret_cast<const unsigned *>(scores + U.kv_row0);
    if (k == (unsigned)(hi - lo)) {
        for (int j = lo + tid; j < hi; j += kT) out[P.sinks + j - lo] = j;
        return;
    }

    // ---- radix select of theta, the bit pattern of the k-th largest candidate
    unsigned prefix = 0, mask = 0, remaining = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kT) sm.hist[i] = 0;
        __syncthreads();
        for (int j0 = lo + tid; j0 < hi; j0 += kT * kLoads) {
            unsigned kk[kLoads];
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const int j = j0 + q * kT;
                kk[q] = j < hi ? sel_key<kCoherent>(keys + j) : 0u;
            }
#pragma unroll
            for (int q = 0; q < kLoads; ++q)
                if (j0 + q * kT < hi && (kk[q] & mask) == prefix)
                    atomicAdd(&sm.hist[(kk[q] >> shift) & 255u], 1u);
        }
        __syncthreads();
        // reverse-order inclusive scan: incl(t) = number of candidates with digit >= 255 - t
        const unsigned h = tid < 256 ? sm.hist[255 - tid] : 0u;
        unsigned tot;
        const unsigned excl = sel_block_scan<kT>(h, sm.warp_sums, &tot);
        const unsigned incl = excl + h;
        if (tid < 256 && incl >= remaining && excl < remaining) {
            sm.scalars[0] = 255u - tid;
            sm.scalars[1] = excl;
        }
        __syncthreads();
        remaining -= sm.scalars[1];
        prefix |= sm.scalars[0] << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    const unsigned theta = prefix, need_eq = remaining;

    // ---- ordered output of the kept middle candidates
    unsigned base_sel = 0, eq_seen = 0;
    for (int c0 = lo; c0 < hi; c0 += kChunk) {
        const int len = min(kChunk, hi - c0);
        __syncthreads();
        {
            unsigned vals[kItems];   // all of the thread's loads in flight together
#pragma unroll
            for (int q = 0; q < kItems; ++q) {
                const int i = tid + q * kT;
                vals[q] = i < len ? sel_key<kCoherent>(keys + c0 + i) : 0u;
            }
#pragma unroll
            for (int q = 0; q < kItems; ++q)
                if (tid + q * kT < len) sm.chunk_keys[tid + q * kT] = vals[q];
        }
        __syncthreads();
        unsigned n_eq = 0;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int i = tid * kItems + it;
            if (i < len && sm.chunk_keys[i] == theta) ++n_eq;
        }
        unsigned eq_total;
        const unsigned eq_before = sel_block_scan<kT>(n_eq, sm.warp_sums, &eq_total);
        unsigned keep_bits = 0, n_keep = 0, eq_rank = eq_seen + eq_before;
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int i = tid * kItems + it;
            if (i >= len) break;
            const unsigned key = sm.chunk_keys[i];
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
        unsigned dst = base_sel + sel_block_scan<kT>(n_keep, sm.warp_sums, &keep_total);
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            if (keep_bits & (1u << it)) {
                if (in_range(P.sinks + dst, b - P.w, status))
                    out[P.sinks + dst] = c0 + tid * kItems + it;
                ++dst;
            }
        }
        base_sel += keep_total;
        eq_seen += eq_total;
    }
}

}  // namespace kvevict
