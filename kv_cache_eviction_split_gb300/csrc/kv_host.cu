// kv_host.cu -- kv_evict_host: the whole eviction path for inputs and outputs in
// host memory, layer groups pipelined against their copies.
//
// The layers are taken in groups of plan->group_layers.  Group g's window
// queries, K and V are copied in on one stream while group g-1 is scored,
// selected and compacted on the caller's stream and group g-2's kept indices
// and rows are copied out on a third, through two device slots that the
// caller's workspace holds (so device memory holds two groups, not the whole
// problem).  Each group is a sub-problem of Lg layers over the same requests:
// its units are (r, l0..l1-1, h), and for every request r those units are one
// contiguous run of the standard unit order, so a group's outputs go back to
// the host as one copy per request straight into their final place.  One
// cudaMemcpyAsync per copy; no batched copies.
//
// Device status does not survive the next group's calls (each zeroes its
// workspace word), so after a group's work its two status words are copied
// (device to device, in stream order) into a per-group array of the
// workspace, read once at the end.
#include <algorithm>
#include <vector>

#include "kv_internal.cuh"
#include "kv_trace.cuh"

using namespace kvevict;

namespace {

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Everything the call derives from the problem and the plan on the host.
struct HostLayout {
    int R, L, H, Hq, d, w, G;          // G: number of groups
    int Lg;                             // layers of the largest group
    long long N;                        // packed tokens
    std::vector<int> l0;                // first layer of each group (G + 1 entries)
    std::vector<long long> rows;        // kept rows of each group
    long long rows_max;
    size_t score_ws, select_ws;         // workspace bytes of the largest sub-problem
    // slot carve-up (bytes from the slot base)
    size_t o_q, o_k, o_v, o_scores, o_pooled, o_sws, o_selws, o_hb, o_ho, o_sel, o_kout,
        o_vout, slot_bytes;
    // shared areas (bytes from the workspace base)
    size_t o_tables, o_headoffs, o_status, total;
    std::vector<size_t> tab_b, tab_o, tab_ho;   // per-group offsets into the shared areas
};

kv_problem sub_problem(const kv_problem *p, int layers) {
    kv_problem s = *p;
    s.num_layers = layers;
    return s;
}

kv_status plan_layout(const kv_problem *p, const kv_host_plan *plan, const int32_t *budgets,
                      HostLayout *Ly) {
    if (!p || !plan) return KV_ERR_INVALID_ARG;
    size_t bytes = 0;
    kv_status st = kv_score_workspace_size(p, &bytes);   // validates the problem
    if (st != KV_OK) return st;
    const int L = p->num_layers;
    if (plan->group_layers < 1 || plan->group_layers > L) return KV_ERR_INVALID_ARG;
    if (plan->pool_kernel < 1 || plan->pool_kernel > 255 || plan->pool_kernel % 2 == 0)
        return KV_ERR_INVALID_ARG;
    if (plan->fused && (plan->pool_kernel > 1 || plan->head_budgets)) return KV_ERR_INVALID_ARG;
    Ly->R = p->num_requests;
    Ly->L = L;
    Ly->H = p->num_kv_heads;
    Ly->Hq = p->num_q_heads;
    Ly->d = p->head_dim;
    Ly->w = p->window;
    Ly->N = Ly->R > 0 ? p->seq_offsets_host[Ly->R] : 0;
    Ly->l0.clear();
    for (int l = 0; l < L; l += plan->group_layers) Ly->l0.push_back(l);
    Ly->G = (int)Ly->l0.size();
    Ly->l0.push_back(L);
    Ly->Lg = std::min(plan->group_layers, L);
    // kept rows per group (the per-layer totals do not change with per-head budgets)
    Ly->rows.assign(Ly->G, 0);
    Ly->rows_max = 0;
    const int R = Ly->R, H = Ly->H;
    for (int g = 0; g < Ly->G; ++g) {
        long long s = 0;
        for (int r = 0; r < R; ++r)
            for (int l = Ly->l0[g]; l < Ly->l0[g + 1]; ++l)
                for (int h = 0; h < H; ++h) s += budgets ? budgets[((long long)r * L + l) * H + h] : 0;
        Ly->rows[g] = s;
        Ly->rows_max = std::max(Ly->rows_max, s);
    }
    // workspaces for the largest need over the group shapes (at most two: a smaller
    // last group can choose smaller pass-1 splits, and so more partials per unit)
    Ly->score_ws = Ly->select_ws = 0;
    for (int g = 0; g < Ly->G; ++g) {
        const kv_problem sub = sub_problem(p, Ly->l0[g + 1] - Ly->l0[g]);
        size_t a = 0, b = 0;
        if ((st = kv_score_workspace_size(&sub, &a)) != KV_OK) return st;
        if ((st = kv_select_workspace_size(&sub, &b)) != KV_OK) return st;
        Ly->score_ws = std::max(Ly->score_ws, a);
        Ly->select_ws = std::max(Ly->select_ws, b);
    }
    const size_t Lg = Ly->Lg, N = (size_t)Ly->N, d = Ly->d;
    const size_t units_g = (size_t)R * Lg * H;
    size_t off = 0;
    auto take = [&](size_t b) {
        const size_t o = off;
        off = round_up(off + b, 256);
        return o;
    };
    Ly->o_q = take((size_t)R * Lg * Ly->Hq * Ly->w * d * 2);
    Ly->o_k = take(Lg * H * N * d * 2);
    Ly->o_v = take(Lg * H * N * d * 2);
    Ly->o_scores = take(Lg * H * N * 4);
    Ly->o_pooled = take(plan->pool_kernel > 1 ? Lg * H * N * 4 : 0);
    Ly->o_sws = take(std::max<size_t>(Ly->score_ws, kHeaderBytes));
    Ly->o_selws = take(std::max<size_t>(Ly->select_ws, kHeaderBytes));
    Ly->o_hb = take(plan->head_budgets ? units_g * 4 : 0);
    Ly->o_ho = take(plan->head_budgets ? (units_g + 1) * 8 : 0);
    const size_t rows = (size_t)std::max<long long>(Ly->rows_max, 1);
    Ly->o_sel = take(rows * 4);
    Ly->o_kout = take(rows * d * 2);
    Ly->o_vout = take(rows * d * 2);
    Ly->slot_bytes = off;
    off = 2 * Ly->slot_bytes;
    // per-group budgets and offsets, uploaded once; per-group head offsets; status words
    Ly->tab_b.clear();
    Ly->tab_o.clear();
    Ly->tab_ho.clear();
    size_t tb = 0;
    std::vector<size_t> ub(Ly->G);
    for (int g = 0; g < Ly->G; ++g) {
        const size_t u = (size_t)R * (Ly->l0[g + 1] - Ly->l0[g]) * H;
        Ly->tab_b.push_back(tb);
        tb = round_up(tb + u * 4, 256);
        Ly->tab_o.push_back(tb);
        tb = round_up(tb + (u + 1) * 8, 256);
        ub[g] = u;
    }
    Ly->o_tables = take(tb);
    size_t th = 0;
    for (int g = 0; g < Ly->G; ++g) {
        Ly->tab_ho.push_back(th);
        th = round_up(th + (plan->head_budgets ? (ub[g] + 1) * 8 : 0), 256);
    }
    Ly->o_headoffs = take(th);
    Ly->o_status = take((size_t)Ly->G * 2 * sizeof(int32_t));
    Ly->total = off;
    return KV_OK;
}

// Streams and events of one call, released on every return path.
struct Streams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
    bool ok = false;
    Streams() {
        ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess;
        for (int i = 0; i < 2 && ok; ++i)
            ok = cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    }
    ~Streams() {
        if (in) cudaStreamSynchronize(in);
        if (out) cudaStreamSynchronize(out);
        for (int i = 0; i < 2; ++i) {
            if (ev_in[i]) cudaEventDestroy(ev_in[i]);
            if (ev_comp[i]) cudaEventDestroy(ev_comp[i]);
            if (ev_out[i]) cudaEventDestroy(ev_out[i]);
        }
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};

}  // namespace

extern "C" {

kv_status kv_evict_host_workspace_size(const kv_problem *p, const kv_host_plan *plan,
                                       const int32_t *budgets_host, size_t *bytes) {
    if (!bytes) return KV_ERR_INVALID_ARG;
    if (p && p->num_requests > 0 && !budgets_host) return KV_ERR_INVALID_ARG;
    HostLayout Ly;
    kv_status st = plan_layout(p, plan, budgets_host, &Ly);
    if (st != KV_OK) return st;
    *bytes = Ly.total;
    return KV_OK;
}

kv_status kv_evict_host(const kv_problem *p, const kv_host_plan *plan, const void *q_win_host,
                        const void *k_host, const void *v_host, const int32_t *budgets_host,
                        int64_t *offsets_host, int32_t *sel_idx_host, void *k_out_host,
                        void *v_out_host, void *workspace, size_t workspace_bytes, void *stream,
                        int32_t *device_status) {
    KV_API_RANGE();
    if (!device_status) return KV_ERR_INVALID_ARG;
    *device_status = KV_OK;
    if (p && p->num_requests > 0 && !budgets_host) return KV_ERR_INVALID_ARG;
    HostLayout Ly;
    kv_status st = plan_layout(p, plan, budgets_host, &Ly);
    if (st != KV_OK) return st;
    if (!offsets_host) return KV_ERR_INVALID_ARG;
    // global offsets (standard unit order); checks every budget
    if ((st = kv_make_offsets(p, budgets_host, offsets_host)) != KV_OK) return st;
    const int R = Ly.R, L = Ly.L, H = Ly.H;
    const long long units = (long long)R * L * H;
    if (units == 0) return KV_OK;
    const long long total_rows = offsets_host[units];
    if (!q_win_host || !k_host || !v_host || !workspace) return KV_ERR_INVALID_ARG;
    if (total_rows > 0 && (!sel_idx_host || !k_out_host || !v_out_host)) return KV_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return KV_ERR_INVALID_ARG;
    if (workspace_bytes < Ly.total) return KV_ERR_WORKSPACE;

    char *ws = static_cast<char *>(workspace);
    cudaStream_t s_comp = (cudaStream_t)stream;
    const size_t d = Ly.d, N = (size_t)Ly.N;
    const size_t row_bytes = d * 2;
    const size_t kv_layer = (size_t)H * N * d * 2;            // bytes of one layer of K (or V)
    const size_t q_layer = (size_t)Ly.Hq * Ly.w * d * 2;      // one (request, layer) of q_win

    // per-group budget and offset tables, built on the host and uploaded once
    std::vector<char> tables(Ly.o_headoffs - Ly.o_tables, 0);
    for (int g = 0; g < Ly.G; ++g) {
        int32_t *b = reinterpret_cast<int32_t *>(tables.data() + Ly.tab_b[g]);
        int64_t *o = reinterpret_cast<int64_t *>(tables.data() + Ly.tab_o[g]);
        long long i = 0, run = 0;
        o[0] = 0;
        for (int r = 0; r < R; ++r)
            for (int l = Ly.l0[g]; l < Ly.l0[g + 1]; ++l)
                for (int h = 0; h < H; ++h, ++i) {
                    b[i] = budgets_host[((long long)r * L + l) * H + h];
                    run += b[i];
                    o[i + 1] = run;
                }
    }
    Streams S;
    if (!S.ok) return KV_ERR_CUDA;
    kv_status result = KV_OK;
    auto cu = [&](cudaError_t e) {
        if (e != cudaSuccess && result == KV_OK) result = KV_ERR_CUDA;
        return e == cudaSuccess;
    };
    cu(cudaMemcpyAsync(ws + Ly.o_tables, tables.data(), tables.size(), cudaMemcpyHostToDevice,
                       s_comp));
    cu(cudaMemsetAsync(ws + Ly.o_status, 0, (size_t)Ly.G * 2 * sizeof(int32_t), s_comp));
    // the slots start free: nothing to wait for in the first two groups
    for (int i = 0; i < 2; ++i) {
        cu(cudaEventRecord(S.ev_comp[i], s_comp));
        cu(cudaEventRecord(S.ev_out[i], s_comp));
    }
    for (int g = 0; g < Ly.G && result == KV_OK; ++g) {
        const int l0 = Ly.l0[g], Lg = Ly.l0[g + 1] - l0, b = g & 1;
        char *slot = ws + b * Ly.slot_bytes;
        const kv_problem sub = sub_problem(p, Lg);
        void *q = slot + Ly.o_q, *k = slot + Ly.o_k, *v = slot + Ly.o_v;
        float *scores = reinterpret_cast<float *>(slot + Ly.o_scores);
        float *pooled = reinterpret_cast<float *>(slot + Ly.o_pooled);
        void *sws = slot + Ly.o_sws, *selws = slot + Ly.o_selws;
        int32_t *sel = reinterpret_cast<int32_t *>(slot + Ly.o_sel);
        void *kout = slot + Ly.o_kout, *vout = slot + Ly.o_vout;
        const int32_t *bud = reinterpret_cast<const int32_t *>(ws + Ly.o_tables + Ly.tab_b[g]);
        const int64_t *offs = reinterpret_cast<const int64_t *>(ws + Ly.o_tables + Ly.tab_o[g]);
        // copy in (after the slot's previous group finished computing)
        cu(cudaStreamWaitEvent(S.in, S.ev_comp[b], 0));
        for (int r = 0; r < R; ++r)
            cu(cudaMemcpyAsync(static_cast<char *>(q) + (size_t)r * Lg * q_layer,
                               static_cast<const char *>(q_win_host) +
                                   ((size_t)r * L + l0) * q_layer,
                               (size_t)Lg * q_layer, cudaMemcpyHostToDevice, S.in));
        cu(cudaMemcpyAsync(k, static_cast<const char *>(k_host) + (size_t)l0 * kv_layer,
                           (size_t)Lg * kv_layer, cudaMemcpyHostToDevice, S.in));
        cu(cudaMemcpyAsync(v, static_cast<const char *>(v_host) + (size_t)l0 * kv_layer,
                           (size_t)Lg * kv_layer, cudaMemcpyHostToDevice, S.in));
        cu(cudaEventRecord(S.ev_in[b], S.in));
        // compute (after the copy in, and after the slot's previous outputs left)
        cu(cudaStreamWaitEvent(s_comp, S.ev_in[b], 0));
        cu(cudaStreamWaitEvent(s_comp, S.ev_out[b], 0));
        if (result != KV_OK) break;
        const long long rows = Ly.rows[g];
        kv_status k_st;
        if (plan->fused) {
            k_st = kv_evict_fused(&sub, q, k, v, bud, offs, rows, scores, sel, kout, vout, sws,
                                  Ly.score_ws, s_comp);
        } else {
            k_st = kv_score(&sub, q, k, v, scores, sws, Ly.score_ws, s_comp);
            const float *ranked = scores;
            if (k_st == KV_OK && plan->pool_kernel > 1) {
                k_st = kv_pool_scores(&sub, plan->pool_kernel, scores, pooled, s_comp);
                ranked = pooled;
            }
            const int32_t *sb = bud;
            const int64_t *so = offs;
            if (k_st == KV_OK && plan->head_budgets) {
                int32_t *hb = reinterpret_cast<int32_t *>(slot + Ly.o_hb);
                int64_t *ho = reinterpret_cast<int64_t *>(slot + Ly.o_ho);
                k_st = kv_head_budgets(&sub, ranked, bud, offs, hb, ho, selws, Ly.select_ws,
                                       s_comp);
                sb = hb;
                so = ho;
                // keep this group's offsets for the host table (device to device)
                const size_t nb = ((size_t)R * Lg * H + 1) * sizeof(int64_t);
                if (k_st == KV_OK)
                    cu(cudaMemcpyAsync(ws + Ly.o_headoffs + Ly.tab_ho[g], ho, nb,
                                       cudaMemcpyDeviceToDevice, s_comp));
            }
            if (k_st == KV_OK)
                k_st = kv_select_topk(&sub, ranked, sb, so, sel, selws, Ly.select_ws, s_comp);
            if (k_st == KV_OK)
                k_st = kv_compact(&sub, k, v, sel, so, rows, kout, vout, s_comp);
        }
        if (k_st != KV_OK) {
            result = k_st;
            break;
        }
        // this group's device status, kept past the next group's calls
        int32_t *stat = reinterpret_cast<int32_t *>(ws + Ly.o_status) + 2 * g;
        cu(cudaMemcpyAsync(stat, sws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s_comp));
        if (!plan->fused)
            cu(cudaMemcpyAsync(stat + 1, selws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                               s_comp));
        cu(cudaEventRecord(S.ev_comp[b], s_comp));
        // copy out: per request, the group's rows are one run of the standard order,
        // where the input budgets put it (per-head budgets keep every (request, layer)
        // total, so they move rows only inside the run)
        cu(cudaStreamWaitEvent(S.out, S.ev_comp[b], 0));
        long long src = 0;
        for (int r = 0; r < R && rows > 0; ++r) {
            const long long u0 = ((long long)r * L + l0) * H;
            const long long dst = offsets_host[u0];
            const long long n = offsets_host[u0 + (long long)Lg * H] - dst;
            if (n > 0) {
                cu(cudaMemcpyAsync(sel_idx_host + dst, sel + src, (size_t)n * 4,
                                   cudaMemcpyDeviceToHost, S.out));
                cu(cudaMemcpyAsync(static_cast<char *>(k_out_host) + dst * row_bytes,
                                   static_cast<char *>(kout) + src * row_bytes,
                                   (size_t)n * row_bytes, cudaMemcpyDeviceToHost, S.out));
                cu(cudaMemcpyAsync(static_cast<char *>(v_out_host) + dst * row_bytes,
                                   static_cast<char *>(vout) + src * row_bytes,
                                   (size_t)n * row_bytes, cudaMemcpyDeviceToHost, S.out));
            }
            src += n;
        }
        cu(cudaEventRecord(S.ev_out[b], S.out));
    }
    // everything issued has finished before the streams go and before the status is read
    const bool synced = cudaStreamSynchronize(S.in) == cudaSuccess &&
                        cudaStreamSynchronize(S.out) == cudaSuccess &&
                        cudaStreamSynchronize(s_comp) == cudaSuccess;
    if (!synced && result == KV_OK) result = KV_ERR_CUDA;
    if (result != KV_OK) return result;
    std::vector<int32_t> stat((size_t)Ly.G * 2);
    if (cudaMemcpy(stat.data(), ws + Ly.o_status, stat.size() * sizeof(int32_t),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return KV_ERR_CUDA;
    for (int32_t c : stat)
        if (c != 0) {
            *device_status = c;
            break;
        }
    if (plan->head_budgets) {
        // the global offsets from each group's per-head offsets
        std::vector<char> ho(Ly.o_status - Ly.o_headoffs);
        if (cudaMemcpy(ho.data(), ws + Ly.o_headoffs, ho.size(), cudaMemcpyDeviceToHost) !=
            cudaSuccess)
            return KV_ERR_CUDA;
        for (int g = 0; g < Ly.G; ++g) {
            const int l0 = Ly.l0[g], Lg = Ly.l0[g + 1] - l0;
            const int64_t *o = reinterpret_cast<const int64_t *>(ho.data() + Ly.tab_ho[g]);
            long long i = 0;
            for (int r = 0; r < R; ++r) {
                const long long u0 = ((long long)r * L + l0) * H;
                const long long base = offsets_host[u0] - o[i];
                for (int j = 0; j < Lg * H; ++j, ++i) offsets_host[u0 + j] = base + o[i];
            }
        }
    }
    return KV_OK;
}

}  // extern "C"
