// kv_internal.cuh -- shared definitions of the kvevict CUDA library (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/kvevict.h"

namespace kvevict {

// Largest R = G * w the kernels accept.
constexpr int kMaxRows = 512;
// Keys per split of the pass-1 attention (each split writes one partial): at most
// kSplitKeys, chosen per problem (DevProblem::split_keys).
constexpr int kSplitKeys = 32768;
constexpr int kMinSplitKeys = 4096;
// Work items per SM the split choice aims for, and the SM count it assumes (GB300).
constexpr int kSplitItemsPerSm = 4;
constexpr int kSplitSms = 152;
// Bytes reserved at the start of every workspace for the status word (int32 at
// offset 0); the score workspace also keeps the fused kernel's grid-barrier
// counter and abort word in it (offsets kGridBarOffset and kGridBarOffset + 64).
// The calls that start a sequence on a workspace zero the status word in-stream
// before their first kernel (kv_score_attention, kv_evict_fused,
// kv_select_topk, kv_head_budgets); kv_score_rescore keeps adding to the word of
// the kv_score_attention it follows.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kGridBarOffset = 64;

// Keys per pass-2 work item (64 tiles of 128 keys).
constexpr int kPass2BlockKeys = 8192;
// Runs of equal-length requests the work-item order tables hold (more: the plan
// tables in the workspace).
constexpr int kMaxOrderRuns = 32;

// Order of the work items of one pass, built on the host (build_item_order) and
// passed to the kernels as a __grid_constant__ parameter, which the item decode
// indexes in place.  An item is one key block (block_keys keys) of one unit.
// Consecutive requests of one length form a run (one run when all lengths are
// equal).  The full blocks come first, unit-major; then the partial last blocks,
// run by run, the runs with the longest partial block first.  A persistent grid
// takes items round-robin, so the equal full blocks fill whole rounds and the
// short partial blocks even out the last ones (the plain unit-major order left
// one SM in ten with 10% more pass-1 work on the ragged batch).
struct ItemOrder {
    int nrun;                            // runs in the tables; 0: not used (plan tables)
    int n_part;                          // runs with a partial last block
    long long full_end;                  // items [0, full_end) are full blocks
    long long unit0[kMaxOrderRuns];      // first unit of run i
    long long full_first[kMaxOrderRuns]; // first full item of run i
    int full_cnt[kMaxOrderRuns];         // full blocks of each unit of run i
    int part_run[kMaxOrderRuns];         // runs with a partial block, longest first
    long long part_first[kMaxOrderRuns]; // first partial item (minus full_end) of part_run[k]
};

// Problem description passed by value to every kernel.
struct DevProblem {
    int R, L, H, Hq, G, d, w, sinks;
    int rule;                 // kv_score_rule
    int rows;                 // G * w
    int max_n;                // longest request
    int split_keys;           // keys per pass-1 split (a power of two, 4096..32768)
    int max_splits;           // ceil(max_n / split_keys)
    long long N_tot;          // packed tokens
    long long units;          // R * L * H
    const long long *cu;      // device cu_seqlens [R + 1]
    const long long *host_cu; // host copy (host code only; never read on the device)
    float scale_log2;         // softmax_scale * log2(e)
    unsigned long long wait_ns;   // limit of the pipeline waits (kv_set_wait_limit_ns)
};

// Limit of the waits for a kernel's own copies and MMAs in flight before it exits.
constexpr unsigned long long kDrainNs = 2000000000ull;

struct UnitInfo {
    int r, l, h;
    int n;
    long long tok0;           // first packed token of the request
    long long kv_row0;        // first row of this unit in K/V/scores ([L][H][N_tot])
    long long q_row0;         // first row of this unit's G*w query rows in q_win
};

__host__ __device__ inline UnitInfo unit_info(const DevProblem &P, long long u, const long long *cu) {
    UnitInfo U;
    U.h = (int)(u % P.H);
    U.l = (int)((u / P.H) % P.L);
    U.r = (int)(u / ((long long)P.H * P.L));
    U.tok0 = cu[U.r];
    U.n = (int)(cu[U.r + 1] - U.tok0);
    U.kv_row0 = ((long long)U.l * P.H + U.h) * P.N_tot + U.tok0;
    U.q_row0 = (((long long)U.r * P.L + U.l) * P.Hq + (long long)U.h * P.G) * P.w;
    return U;
}

// Unit and block of item g of a pass ordered by O (O.nrun > 0).  Item counts stay
// below 2^31 (the row limits of make_problem), so the arithmetic is 32-bit.  Not
// inlined: it runs once per work item, and inlined into every role's item loop it
// took registers from the kernels' tile loops.
static __device__ __noinline__ void order_decode(const ItemOrder &O, long long g64, long long &u,
                                                 int &blk) {
    const int g = (int)g64;
    if (g64 < O.full_end) {
        int r = 0;
        while (r + 1 < O.nrun && O.full_first[r + 1] <= g64) ++r;
        const int off = g - (int)O.full_first[r];
        u = O.unit0[r] + off / O.full_cnt[r];
        blk = off % O.full_cnt[r];
    } else {
        const int j = g - (int)O.full_end;
        int k = 0;
        while (k + 1 < O.n_part && O.part_first[k + 1] <= j) ++k;
        const int r = O.part_run[k];
        u = O.unit0[r] + (j - (int)O.part_first[k]);
        blk = O.full_cnt[r];
    }
}

// Score workspace carve-up (all offsets 256-byte aligned).
struct ScoreWs {
    int *status;
    float2 *part_ml;          // [units][max_splits * parts][rows]  (m in log2 units, l)
    float *part_o;            // [units][max_splits * parts][rows][d]
    float2 *stat_ml;          // [units][rows]  merged (m, l)
    float *stat_a2;           // [units][rows]  ||a_hi + a_lo||^2
    __nv_bfloat16 *a_hi;      // [units][a_rows][d]  bf16(a)
    __nv_bfloat16 *a_lo;      // [units][a_rows][d]  bf16(a - a_hi); rows >= rows are zero
    int32_t *plan;            // [units + 1] work plan of the pass being launched
    int32_t *plan2;           // [units + 1] pass-2 plan of the fused kernel (both live)
    float *part_scores;       // [chunks][L*H*N_tot] when chunks > 1
    float *v2;                // [L*H*N_tot] ||v_j||^2 of every key (written by pass 1)
    int a_rows;               // chunks * 128
    int chunks;               // ceil(rows / 128)
    int parts;                // pass-1 partials per split: 2 with one chunk, else 1
    size_t total;
};

ScoreWs score_ws_layout(const DevProblem &P, void *base);

// The item order of a pass with key blocks of `block_keys` keys (from host_cu);
// nrun = 0 when the requests form more than kMaxOrderRuns runs of one length.
void build_item_order(const DevProblem &P, long long block_keys, ItemOrder *O);
// plan[u] = sum over units u' < u of ceil(n_u' / keys_per_block); plan[units] = total.
void launch_plan(const DevProblem &P, int keys_per_block, int32_t *plan, cudaStream_t s);
// 2-D TMA map over a row-major [rows][D] bf16 tensor: box 128 rows x 64 columns,
// 128-byte swizzle, out-of-range rows read as zero.  False if encoding fails.
bool make_tile_map(CUtensorMap *m, const void *base, long long rows, int D);
// Total blocks of ceil(n_u / keys_per_block) over all units (host, from host_cu).
long long total_blocks(const DevProblem &P, int keys_per_block);

// Launchers (return cudaGetLastError() of their launches).
cudaError_t launch_attention_partials(const DevProblem &P, const __nv_bfloat16 *q,
                                      const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                      const ScoreWs &ws, cudaStream_t s);
cudaError_t launch_attention(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                             const __nv_bfloat16 *v, const ScoreWs &ws, cudaStream_t s);
cudaError_t launch_rescore(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                           const __nv_bfloat16 *v, float *scores, const ScoreWs &ws,
                           cudaStream_t s);
cudaError_t launch_pool(const DevProblem &P, int kernel, const float *in, float *out,
                        cudaStream_t s);
cudaError_t launch_block_sum(const DevProblem &P, int block_layers, const float *scores,
                             float *out, cudaStream_t s);
cudaError_t launch_compact_blocks(const DevProblem &P, int block_layers, const __nv_bfloat16 *k,
                                  const __nv_bfloat16 *v, const int32_t *block_sel,
                                  const int64_t *block_offsets, const int64_t *offsets,
                                  long long total_rows, __nv_bfloat16 *kout,
                                  __nv_bfloat16 *vout, cudaStream_t s);
// Scratch bytes of the per-head budget select (after the status header).
size_t head_budget_ws_bytes(const DevProblem &P);
cudaError_t launch_head_budgets(const DevProblem &P, const float *scores, const int32_t *budgets,
                                const int64_t *offsets, int32_t *budgets_out,
                                int64_t *offsets_out, int *status, void *scratch,
                                cudaStream_t s);
cudaError_t launch_select(const DevProblem &P, const float *scores, const int32_t *budgets,
                          const int64_t *offsets, int32_t *sel, int *status, cudaStream_t s);
cudaError_t launch_compact(const DevProblem &P, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                           const int32_t *sel, const int64_t *offsets, long long total_rows,
                           __nv_bfloat16 *kout, __nv_bfloat16 *vout, cudaStream_t s);
// Score -> select -> compaction in one cooperative launch (kv_fused.cu); the
// select's status goes to the score workspace's status word.
cudaError_t launch_fused(const DevProblem &P, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                         const __nv_bfloat16 *v, const int32_t *budgets, const int64_t *offsets,
                         long long total_rows, float *scores, int32_t *sel, __nv_bfloat16 *kout,
                         __nv_bfloat16 *vout, const ScoreWs &ws, cudaStream_t s);

__device__ inline void post_status(int *status, int code) {
    atomicCAS(status, 0, code);
}

// Bounds checks of the debug build (-DKV_DEBUG_BOUNDS, libkvevict_debug.so): every
// TMA tile coordinate, workspace offset and gather index is tested against the
// extent of its tensor before use.  in_range(i, n, status) is true when
// 0 <= i < n; otherwise it posts KV_ERR_INVALID_ARG and the caller skips the
// access (a pipeline producer instead stops issuing and aborts its CTA's pipeline,
// whose other roles drain out as after an expired wait).  Nothing traps.  Calls
// without a status word (kv_compact has no workspace) pass nullptr and only skip.
// In the release build it is the constant true and costs nothing.
#ifdef KV_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif
__device__ __forceinline__ bool in_range(long long i, long long n, int *status) {
    if constexpr (!kDebugBounds) {
        return true;
    } else {
        const bool ok = i >= 0 && i < n;
        if (!ok && status) post_status(status, KV_ERR_INVALID_ARG);
        return ok;
    }
}
// Rows of the packed K/V (and scores, ||v||^2) tensors, and of the window queries.
__host__ __device__ inline long long kv_rows_total(const DevProblem &P) {
    return (long long)P.L * P.H * P.N_tot;
}
__host__ __device__ inline long long q_rows_total(const DevProblem &P) {
    return (long long)P.R * P.L * P.Hq * P.w;
}

}  // namespace kvevict
