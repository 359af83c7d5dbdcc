// kv_api.cu -- the extern "C" entry points: argument checks, workspace carve-up,
// launches, the offsets scan and the per-layer budget policies (host code).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "kv_internal.cuh"
#include "kv_trace.cuh"

using namespace kvevict;

namespace {

// Pipeline wait limit of the kernels (kv_set_wait_limit_ns).
std::atomic<unsigned long long> g_wait_ns{2000000000ull};

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace kvevict {

void build_item_order(const DevProblem &P, long long bk, ItemOrder *O) {
    const long long *cu = P.host_cu;
    std::memset(O, 0, sizeof *O);
    if (P.R == 0) return;
    const long long lh = (long long)P.L * P.H;
    // runs of consecutive requests with one length
    std::vector<int> first, count;
    for (int r = 0; r < P.R; ++r) {
        const long long n = cu[r + 1] - cu[r];
        if (r > 0 && n == cu[r] - cu[r - 1]) {
            ++count.back();
        } else {
            first.push_back(r);
            count.push_back(1);
        }
    }
    if ((int)first.size() > kMaxOrderRuns) return;
    const int runs = (int)first.size();
    long long acc = 0;
    std::vector<int> part;
    for (int i = 0; i < runs; ++i) {
        const long long n = cu[first[i] + 1] - cu[first[i]];
        O->unit0[i] = first[i] * lh;
        O->full_first[i] = acc;
        O->full_cnt[i] = (int)(n / bk);
        acc += count[i] * lh * (n / bk);
        if (n % bk) part.push_back(i);
    }
    O->full_end = acc;
    auto part_len = [&](int i) { return (cu[first[i] + 1] - cu[first[i]]) % bk; };
    std::stable_sort(part.begin(), part.end(),
                     [&](int a, int b) { return part_len(a) > part_len(b); });
    long long pacc = 0;
    for (size_t k = 0; k < part.size(); ++k) {
        O->part_run[k] = part[k];
        O->part_first[k] = pacc;
        pacc += count[part[k]] * lh;
    }
    O->n_part = (int)part.size();
    O->nrun = runs;
}

}  // namespace kvevict

namespace {

// Validates the problem description and fills the device-side copy.
kv_status make_problem(const kv_problem *p, DevProblem *P) {
    if (!p) return KV_ERR_INVALID_ARG;
    if (p->num_requests < 0 || p->num_layers < 1 || p->num_kv_heads < 1 ||
        p->num_q_heads < p->num_kv_heads || p->num_q_heads % p->num_kv_heads != 0 ||
        p->window < 1 || p->num_sinks < 0 || p->score_rule < KV_SCORE_DROPKV ||
        p->score_rule > KV_SCORE_ATTN_SUM)
        return KV_ERR_INVALID_ARG;
    if (!(p->softmax_scale > 0.0f) || !std::isfinite(p->softmax_scale)) return KV_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return KV_ERR_UNSUPPORTED;
    const long long G = p->num_q_heads / p->num_kv_heads;
    if (G * p->window > kMaxRows) return KV_ERR_UNSUPPORTED;
    P->R = p->num_requests;
    P->L = p->num_layers;
    P->H = p->num_kv_heads;
    P->Hq = p->num_q_heads;
    P->G = (int)G;
    P->d = p->head_dim;
    P->w = p->window;
    P->sinks = p->num_sinks;
    P->rule = p->score_rule;
    P->rows = (int)(G * p->window);
    P->cu = reinterpret_cast<const long long *>(p->seq_offsets_dev);
    P->host_cu = reinterpret_cast<const long long *>(p->seq_offsets_host);
    P->scale_log2 = p->softmax_scale * 1.4426950408889634f;
    P->wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    P->units = (long long)P->R * P->L * P->H;
    P->max_n = 0;
    P->N_tot = 0;
    if (P->R > 0) {
        if (!p->seq_offsets_host || !p->seq_offsets_dev) return KV_ERR_INVALID_ARG;
        if (p->seq_offsets_host[0] != 0) return KV_ERR_INVALID_ARG;
        for (int r = 0; r < P->R; ++r) {
            const long long n = p->seq_offsets_host[r + 1] - p->seq_offsets_host[r];
            if (n < (long long)p->num_sinks + p->window || n < 1 || n >= (1LL << 31))
                return KV_ERR_INVALID_ARG;
            P->max_n = std::max<long long>(P->max_n, n);
        }
        P->N_tot = p->seq_offsets_host[P->R];
    }
    // TMA tile coordinates are 32-bit: the packed K/V rows, the window query rows
    // and pass 2's rows of a must each stay below 2^31.
    const long long kRowLimit = 1LL << 31;
    if ((long long)P->L * P->H * P->N_tot >= kRowLimit ||
        (long long)P->R * P->L * P->Hq * P->w >= kRowLimit ||
        P->units * (long long)((P->rows + 127) / 128 * 128) >= kRowLimit)
        return KV_ERR_UNSUPPORTED;
    // Splits of kSplitKeys keys, halved (down to kMinSplitKeys) while the pass-1 work items
    // -- splits over all units times the row-chunk pairs -- would leave fewer than
    // kSplitItemsPerSm per SM: with one split per unit, the last round of a persistent
    // grid runs part-empty.  The choice depends on the shapes only, so workspace sizes
    // are known on the host.
    const int chunks = (P->rows + 127) / 128;
    const long long pairs = chunks == 1 ? 1 : (chunks + 1) / 2;
    auto items = [&](long long split) {
        long long per_layer_head = 0;
        for (int r = 0; r < P->R; ++r) {
            const long long n = p->seq_offsets_host[r + 1] - p->seq_offsets_host[r];
            per_layer_head += (n + split - 1) / split;
        }
        return per_layer_head * P->L * P->H * pairs;
    };
    P->split_keys = kSplitKeys;
    while (P->split_keys > kMinSplitKeys &&
           items(P->split_keys) < (long long)kSplitItemsPerSm * kSplitSms)
        P->split_keys /= 2;
    P->max_splits = (int)((P->max_n + P->split_keys - 1) / P->split_keys);
    return KV_OK;
}

kv_status map_cuda(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

}  // namespace

namespace kvevict {

ScoreWs score_ws_layout(const DevProblem &P, void *base) {
    ScoreWs ws{};
    char *b = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *p = b ? b + off : nullptr;
        off = round_up(off + bytes, 256);
        return p;
    };
    const size_t U = (size_t)P.units, S = (size_t)P.max_splits, Rr = (size_t)P.rows, D = P.d;
    ws.chunks = (P.rows + 127) / 128;
    ws.parts = ws.chunks == 1 ? 2 : 1;
    ws.a_rows = ws.chunks * 128;
    const size_t AR = (size_t)ws.a_rows, SP = S * (size_t)ws.parts;
    ws.status = reinterpret_cast<int *>(take(kHeaderBytes));
    ws.part_ml = reinterpret_cast<float2 *>(take(U * SP * Rr * sizeof(float2)));
    ws.part_o = reinterpret_cast<float *>(take(U * SP * Rr * D * sizeof(float)));
    ws.stat_ml = reinterpret_cast<float2 *>(take(U * Rr * sizeof(float2)));
    ws.stat_a2 = reinterpret_cast<float *>(take(U * Rr * sizeof(float)));
    ws.a_hi = reinterpret_cast<__nv_bfloat16 *>(take(U * AR * D * sizeof(__nv_bfloat16)));
    ws.a_lo = reinterpret_cast<__nv_bfloat16 *>(take(U * AR * D * sizeof(__nv_bfloat16)));
    ws.plan = reinterpret_cast<int32_t *>(take((U + 1) * sizeof(int32_t)));
    ws.plan2 = reinterpret_cast<int32_t *>(take((U + 1) * sizeof(int32_t)));
    const size_t keys = (size_t)P.L * P.H * (size_t)P.N_tot;
    ws.part_scores = reinterpret_cast<float *>(
        take(ws.chunks > 1 ? (size_t)ws.chunks * keys * sizeof(float) : 0));
    ws.v2 = reinterpret_cast<float *>(take(keys * sizeof(float)));
    ws.total = off;
    return ws;
}

}  // namespace kvevict

extern "C" {

const char *kv_status_string(kv_status s) {
    switch (s) {
        case KV_OK: return "KV_OK";
        case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
        case KV_ERR_BUDGET: return "KV_ERR_BUDGET";
        case KV_ERR_WORKSPACE: return "KV_ERR_WORKSPACE";
        case KV_ERR_CUDA: return "KV_ERR_CUDA";
        case KV_ERR_TIMEOUT: return "KV_ERR_TIMEOUT";
        case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    }
    return "KV_ERR_UNKNOWN";
}

kv_status kv_score_workspace_size(const kv_problem *p, size_t *bytes) {
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (!bytes) return KV_ERR_INVALID_ARG;
    *bytes = score_ws_layout(P, nullptr).total;
    return KV_OK;
}

static kv_status check_score_args(const kv_problem *p, DevProblem *P, const void *q,
                                  const void *k, const void *v, const void *ws, size_t ws_bytes) {
    kv_status st = make_problem(p, P);
    if (st != KV_OK) return st;
    if (P->units == 0) return KV_OK;
    if (!q || !k || !v || !ws) return KV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(ws)) return KV_ERR_INVALID_ARG;
    if (ws_bytes < score_ws_layout(*P, nullptr).total) return KV_ERR_WORKSPACE;
    return KV_OK;
}

kv_status kv_score_attention(const kv_problem *p, const void *q_win, const void *k, const void *v,
                             void *workspace, size_t workspace_bytes, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = check_score_args(p, &P, q_win, k, v, workspace, workspace_bytes);
    if (st != KV_OK || P.units == 0) return st;
    ScoreWs ws = score_ws_layout(P, workspace);
    // a new scoring sequence: its status word starts at zero (the workspace may be
    // uninitialised memory)
    if (cudaMemsetAsync(ws.status, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess)
        return KV_ERR_CUDA;
    return map_cuda(launch_attention(P, (const __nv_bfloat16 *)q_win, (const __nv_bfloat16 *)k,
                                     (const __nv_bfloat16 *)v, ws, (cudaStream_t)stream));
}

kv_status kv_score_rescore(const kv_problem *p, const void *q_win, const void *k, const void *v,
                           float *scores, void *workspace, size_t workspace_bytes, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = check_score_args(p, &P, q_win, k, v, workspace, workspace_bytes);
    if (st != KV_OK || P.units == 0) return st;
    if (!scores || !aligned16(scores)) return KV_ERR_INVALID_ARG;
    ScoreWs ws = score_ws_layout(P, workspace);
    return map_cuda(launch_rescore(P, (const __nv_bfloat16 *)q_win, (const __nv_bfloat16 *)k,
                                   (const __nv_bfloat16 *)v, scores, ws, (cudaStream_t)stream));
}

kv_status kv_score(const kv_problem *p, const void *q_win, const void *k, const void *v,
                   float *scores, void *workspace, size_t workspace_bytes, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = check_score_args(p, &P, q_win, k, v, workspace, workspace_bytes);
    if (st != KV_OK || P.units == 0) return st;
    if (!scores || !aligned16(scores)) return KV_ERR_INVALID_ARG;
    st = kv_score_attention(p, q_win, k, v, workspace, workspace_bytes, stream);
    if (st != KV_OK) return st;
    return kv_score_rescore(p, q_win, k, v, scores, workspace, workspace_bytes, stream);
}

kv_status kv_pool_scores(const kv_problem *p, int32_t kernel, const float *scores_in,
                         float *scores_out, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (kernel < 1 || kernel > 255 || kernel % 2 == 0) return KV_ERR_INVALID_ARG;
    if (P.units == 0) return KV_OK;
    if (!scores_in || !scores_out || !aligned16(scores_in) || !aligned16(scores_out))
        return KV_ERR_INVALID_ARG;
    const uintptr_t bytes = (uintptr_t)P.L * P.H * (uintptr_t)P.N_tot * sizeof(float);
    const uintptr_t a = reinterpret_cast<uintptr_t>(scores_in);
    const uintptr_t b = reinterpret_cast<uintptr_t>(scores_out);
    if (a < b + bytes && b < a + bytes) return KV_ERR_INVALID_ARG;
    return map_cuda(launch_pool(P, kernel, scores_in, scores_out, (cudaStream_t)stream));
}

kv_status kv_make_offsets(const kv_problem *p, const int32_t *budgets_host, int64_t *offsets_host) {
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (!offsets_host || (P.units > 0 && !budgets_host)) return KV_ERR_INVALID_ARG;
    offsets_host[0] = 0;
    for (long long u = 0; u < P.units; ++u) {
        const int r = (int)(u / ((long long)P.L * P.H));
        const long long n = p->seq_offsets_host[r + 1] - p->seq_offsets_host[r];
        const long long b = budgets_host[u];
        if (b < (long long)P.sinks + P.w || b > n) return KV_ERR_BUDGET;
        offsets_host[u + 1] = offsets_host[u] + b;
    }
    return KV_OK;
}

kv_status kv_select_workspace_size(const kv_problem *p, size_t *bytes) {
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (!bytes) return KV_ERR_INVALID_ARG;
    *bytes = kHeaderBytes + head_budget_ws_bytes(P);
    return KV_OK;
}

kv_status kv_select_topk(const kv_problem *p, const float *scores, const int32_t *budgets_dev,
                         const int64_t *offsets_dev, int32_t *sel_idx, void *workspace,
                         size_t workspace_bytes, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK || P.units == 0) return st;
    if (!scores || !budgets_dev || !offsets_dev || !sel_idx || !workspace) return KV_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(budgets_dev) || !aligned16(offsets_dev) ||
        !aligned16(sel_idx) || !aligned16(workspace))
        return KV_ERR_INVALID_ARG;
    if (workspace_bytes < kHeaderBytes) return KV_ERR_WORKSPACE;
    int *status = static_cast<int *>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess)
        return KV_ERR_CUDA;
    return map_cuda(launch_select(P, scores, budgets_dev, offsets_dev, sel_idx, status,
                                  (cudaStream_t)stream));
}

kv_status kv_head_budgets(const kv_problem *p, const float *scores, const int32_t *budgets_dev,
                          const int64_t *offsets_dev, int32_t *budgets_out_dev,
                          int64_t *offsets_out_dev, void *workspace, size_t workspace_bytes,
                          void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK || P.units == 0) return st;
    if (!scores || !budgets_dev || !offsets_dev || !budgets_out_dev || !offsets_out_dev ||
        !workspace)
        return KV_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(budgets_dev) || !aligned16(offsets_dev) ||
        !aligned16(budgets_out_dev) || !aligned16(offsets_out_dev) || !aligned16(workspace))
        return KV_ERR_INVALID_ARG;
    if (budgets_out_dev == budgets_dev || offsets_out_dev == offsets_dev) return KV_ERR_INVALID_ARG;
    if (workspace_bytes < kHeaderBytes + head_budget_ws_bytes(P)) return KV_ERR_WORKSPACE;
    // the layer-wide counts are 32-bit
    if ((long long)P.H * P.max_n >= (1LL << 32)) return KV_ERR_UNSUPPORTED;
    // a layer whose budgets fail the check is copied through unchanged, so the
    // kv_select_topk that takes these outputs (and zeroes the word again) fails the
    // same check on the same unit and posts KV_ERR_BUDGET once more
    int *status = static_cast<int *>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess)
        return KV_ERR_CUDA;
    return map_cuda(launch_head_budgets(P, scores, budgets_dev, offsets_dev, budgets_out_dev,
                                        offsets_out_dev, status,
                                        static_cast<char *>(workspace) + kHeaderBytes,
                                        (cudaStream_t)stream));
}

kv_status kv_block_scores(const kv_problem *p, int32_t block_layers, const float *scores,
                          float *block_scores, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (block_layers < 1 || P.L % block_layers != 0) return KV_ERR_INVALID_ARG;
    if (P.units == 0) return KV_OK;
    if (!scores || !block_scores || !aligned16(scores) || !aligned16(block_scores))
        return KV_ERR_INVALID_ARG;
    return map_cuda(launch_block_sum(P, block_layers, scores, block_scores, (cudaStream_t)stream));
}

kv_status kv_compact_blocks(const kv_problem *p, int32_t block_layers, const void *k,
                            const void *v, const int32_t *block_sel_idx,
                            const int64_t *block_offsets_dev, const int64_t *offsets_dev,
                            int64_t total_rows, void *k_out, void *v_out, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK || P.units == 0) return st;
    if (block_layers < 1 || P.L % block_layers != 0 || total_rows < 0) return KV_ERR_INVALID_ARG;
    if (total_rows == 0) return KV_OK;
    if (!k || !v || !block_sel_idx || !block_offsets_dev || !offsets_dev || !k_out || !v_out)
        return KV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(block_sel_idx) ||
        !aligned16(block_offsets_dev) || !aligned16(offsets_dev) || !aligned16(k_out) ||
        !aligned16(v_out))
        return KV_ERR_INVALID_ARG;
    return map_cuda(launch_compact_blocks(P, block_layers, (const __nv_bfloat16 *)k,
                                          (const __nv_bfloat16 *)v, block_sel_idx,
                                          block_offsets_dev, offsets_dev, total_rows,
                                          (__nv_bfloat16 *)k_out, (__nv_bfloat16 *)v_out,
                                          (cudaStream_t)stream));
}

kv_status kv_evict_fused(const kv_problem *p, const void *q_win, const void *k, const void *v,
                         const int32_t *budgets_dev, const int64_t *offsets_dev,
                         int64_t total_rows, float *scores, int32_t *sel_idx, void *k_out,
                         void *v_out, void *workspace, size_t workspace_bytes, void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = check_score_args(p, &P, q_win, k, v, workspace, workspace_bytes);
    if (st != KV_OK || P.units == 0) return st;
    if (total_rows < 0 || !scores || !budgets_dev || !offsets_dev || !sel_idx)
        return KV_ERR_INVALID_ARG;
    if (total_rows > 0 && (!k_out || !v_out)) return KV_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(budgets_dev) || !aligned16(offsets_dev) ||
        !aligned16(sel_idx) || (total_rows > 0 && (!aligned16(k_out) || !aligned16(v_out))))
        return KV_ERR_INVALID_ARG;
    ScoreWs ws = score_ws_layout(P, workspace);
    return map_cuda(launch_fused(P, (const __nv_bfloat16 *)q_win, (const __nv_bfloat16 *)k,
                                 (const __nv_bfloat16 *)v, budgets_dev, offsets_dev, total_rows,
                                 scores, sel_idx, (__nv_bfloat16 *)k_out, (__nv_bfloat16 *)v_out,
                                 ws, (cudaStream_t)stream));
}

kv_status kv_compact(const kv_problem *p, const void *k, const void *v, const int32_t *sel_idx,
                     const int64_t *offsets_dev, int64_t total_rows, void *k_out, void *v_out,
                     void *stream) {
    KV_API_RANGE();
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK || P.units == 0) return st;
    if (total_rows < 0) return KV_ERR_INVALID_ARG;
    if (total_rows == 0) return KV_OK;
    if (!k || !v || !sel_idx || !offsets_dev || !k_out || !v_out) return KV_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(sel_idx) || !aligned16(offsets_dev) ||
        !aligned16(k_out) || !aligned16(v_out))
        return KV_ERR_INVALID_ARG;
    return map_cuda(launch_compact(P, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, sel_idx,
                                   offsets_dev, total_rows, (__nv_bfloat16 *)k_out,
                                   (__nv_bfloat16 *)v_out, (cudaStream_t)stream));
}

void kv_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

uint64_t kv_get_wait_limit_ns(void) { return g_wait_ns.load(std::memory_order_relaxed); }

kv_status kv_check_status(void *workspace, void *stream, int32_t *device_status) {
    KV_API_RANGE();
    if (!workspace || !device_status) return KV_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KV_ERR_CUDA;
    if (word != 0 && cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return KV_ERR_CUDA;
    *device_status = word;
    return KV_OK;
}

// ----------------------------------------------------------------------------
// per-layer budgets (host)
// ----------------------------------------------------------------------------
static kv_status largest_remainder(int L, int B, const std::vector<double> &mult, int32_t *out) {
    std::vector<double> x(L), frac(L);
    long long sum = 0;
    for (int l = 0; l < L; ++l) {
        x[l] = (double)B * mult[l];
        const double f = std::floor(x[l]);
        frac[l] = x[l] - f;
        out[l] = (int32_t)f;
        sum += (long long)f;
    }
    const long long deficit = (long long)L * B - sum;
    if (deficit < 0 || deficit > L) return KV_ERR_INVALID_ARG;
    std::vector<int> order(L);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (frac[a] != frac[b]) return frac[a] > frac[b];
        return a < b;
    });
    for (long long i = 0; i < deficit; ++i) out[order[i]] += 1;
    return KV_OK;
}

kv_status kv_budgets_pyramid(int32_t num_layers, int32_t mean_budget, double hi, double lo,
                             double curve, int32_t *budgets_out) {
    if (num_layers < 1 || mean_budget < 0 || !budgets_out || !(hi >= lo) || !(lo >= 0.0) ||
        !(curve > 0.0))
        return KV_ERR_INVALID_ARG;
    const int L = num_layers;
    std::vector<double> m(L, 1.0);
    if (L > 1) {
        double sum = 0.0;
        for (int l = 0; l < L; ++l) {
            m[l] = lo + (hi - lo) * std::pow(1.0 - (double)l / (double)(L - 1), curve);
            sum += m[l];
        }
        const double mean = sum / L;
        if (!(mean > 0.0)) return KV_ERR_INVALID_ARG;
        for (int l = 0; l < L; ++l) m[l] = m[l] / mean;
    }
    return largest_remainder(L, mean_budget, m, budgets_out);
}

kv_status kv_budgets_fraction(const kv_problem *p, double q, int32_t *budgets_host) {
    DevProblem P;
    kv_status st = make_problem(p, &P);
    if (st != KV_OK) return st;
    if (!(q >= 0.0 && q <= 1.0)) return KV_ERR_INVALID_ARG;
    if (P.units > 0 && !budgets_host) return KV_ERR_INVALID_ARG;
    for (long long u = 0; u < P.units; ++u) {
        const int r = (int)(u / ((long long)P.L * P.H));
        const long long n = p->seq_offsets_host[r + 1] - p->seq_offsets_host[r];
        const long long rest = n - P.sinks - P.w;
        budgets_host[u] = (int32_t)(P.sinks + P.w + (long long)std::floor(q * (double)rest));
    }
    return KV_OK;
}

kv_status kv_budgets_ripple(int32_t num_layers, int32_t mean_budget, const double *profile,
                            double beta, double gamma, int32_t *budgets_out) {
    if (num_layers < 1 || mean_budget < 0 || !profile || !budgets_out || !(beta >= 0.0) ||
        !(gamma >= 1.0))
        return KV_ERR_INVALID_ARG;
    const int L = num_layers;
    double smin = profile[0], smax = profile[0];
    for (int l = 0; l < L; ++l) {
        if (!std::isfinite(profile[l])) return KV_ERR_INVALID_ARG;
        smin = std::min(smin, profile[l]);
        smax = std::max(smax, profile[l]);
    }
    std::vector<double> m(L);
    double sum = 0.0;
    for (int l = 0; l < L; ++l) {
        const double shat = (smax == smin) ? 0.0 : (profile[l] - smin) / (smax - smin);
        double t = std::exp(beta * shat);
        if (std::isfinite(gamma)) t = std::min(std::max(t, 1.0 / gamma), gamma);
        m[l] = t;
        sum += t;
    }
    const double mean = sum / L;
    for (int l = 0; l < L; ++l) m[l] = m[l] / mean;
    return largest_remainder(L, mean_budget, m, budgets_out);
}

}  // extern "C"
