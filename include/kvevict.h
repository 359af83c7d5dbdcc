/*
 * kvevict.h -- C ABI of the GB300 KV-cache eviction hot path.
 *
 * Three steps run on one GPU, each asynchronous on the caller's stream:
 *
 *   kv_score        per-token DropKV removal score of every cached key
 *                   (or, by kv_problem.score_rule, its squared form or the
 *                   SnapKV/PyramidKV attention sum)
 *   kv_pool_scores  optional 1-D max pooling of the scores before selection
 *   kv_head_budgets optional per-head budgets from the scores (AdaDropKV)
 *   kv_block_scores, kv_compact_blocks  block eviction (BellowsKV)
 *   kv_select_topk  budgeted per-(request, layer, KV head) selection
 *   kv_compact      ragged gather of the kept K/V rows
 *
 * Definitions (the pages these steps follow):
 *
 *  - Score.  "DropKV: Decoupling Residual-Output Perturbation for Near-Optimal
 *    KV-Cache Eviction", Key Contributions item 1 and "Methodology in Plain
 *    English": deleting token j alone shifts an attention output a by
 *    p_j / (1 - p_j) * ||a - v_j||_2.  Here the score of key j is that shift
 *    summed, unsquared, over the last w query positions of the request (the
 *    observation window) and the G query heads that share the KV head, each
 *    query attending causally.  It is computed in two streaming passes
 *    (window attention with split-K and a merge, then a rescoring pass that
 *    expands ||a - v||^2 = ||a||^2 - 2 a.v + ||v||^2, the expansion the same
 *    section describes), never materialising the n x w attention matrix.
 *  - Other aggregation rules (score_rule).  KV_SCORE_DROPKV_SQUARED: the same
 *    page, "Methodology in Plain English", accumulates the shift over the
 *    window squared: S_j = sum (p_j / (1 - p_j))^2 * ||a - v_j||_2^2.
 *    KV_SCORE_ATTN_SUM: the PyramidKV guide, "Observation Window and
 *    Aggregated Attention Eviction": S_j = sum of the attention weights p_j of
 *    the window queries over queries and heads.  Both sum over the same rows.
 *  - Pooling.  DropKV, "Methodology in Plain English" (a max-pool over
 *    neighbouring scores, after SnapKV; kernel size 11 in its evaluation) and
 *    the BellowsKV blog (the maximum score in a 13-position window centred on
 *    each token).
 *  - Selection.  Same page, "Methodology in Plain English" (keep the highest
 *    scores, pin the recent w) and the PyramidKV guide, "Observation Window
 *    and Aggregated Attention Eviction" (always keep the first 4 sinks).
 *  - Compaction.  GraceKV project page, section 05 "physical cache packing":
 *    each layer-KV-head pair gets a cache of its own length.
 *  - Layer budgets.  RippleKV, Eq. (9)-(12) and PyramidKV guide,
 *    "Layer-Adaptive Dynamic Budget Allocation".
 *
 * Shapes.  R requests with lengths n_r (tokens packed, cu_seqlens
 * seq_offsets[r] .. seq_offsets[r+1]), L layers, H KV heads, H_q = G*H query
 * heads, head dim d in {64, 128}, window w, sinks s.  A "unit" (also
 * "segment") is one (request, layer, KV head); units are ordered request-major,
 * then layer, then head: u = (r*L + l)*H + h.
 *
 * Layouts (row-major; bf16 = IEEE bfloat16):
 *   q_win   bf16 [R][L][H_q][w][d]   queries at positions n_r - w .. n_r - 1
 *   k, v    bf16 [L][H][N_tot][d]    N_tot = seq_offsets[R]
 *   scores  f32  [L][H][N_tot]
 *   budgets i32  [R][L][H]           kept tokens per unit, sinks and window included
 *   offsets i64  [R*L*H + 1]         exclusive scan of budgets (rows)
 *   sel_idx i32  [offsets[R*L*H]]    kept token indices, local to the request, ascending
 *   k_out, v_out bf16 [offsets[R*L*H]][d]
 *
 * Ownership.  The caller allocates and owns every buffer, host or device.
 * The library allocates nothing and keeps no state between calls; the
 * scratch it needs is the caller's workspace, sized by *_workspace_size.
 * Functions are re-entrant; calls that share a workspace must be ordered on
 * one stream.
 *
 * Errors.  Argument checks run on the host before anything is launched and
 * return KV_ERR_INVALID_ARG / KV_ERR_BUDGET / KV_ERR_WORKSPACE /
 * KV_ERR_UNSUPPORTED.  A failed launch returns KV_ERR_CUDA.  Conditions only
 * the device can see (a budget in device memory out of range, an offsets table
 * that disagrees with the budgets, a V value fp16 cannot carry, a bounded wait
 * that expired) are written to a status word in the workspace header;
 * kv_check_status reads it.  A workspace needs no initialisation: its first
 * 256 bytes are a header whose first int32 is the status word, and each call
 * that starts a sequence on the workspace zeroes that word (an in-stream memset
 * before its first kernel): kv_score_attention (so kv_score), kv_evict_fused,
 * kv_select_topk and kv_head_budgets.  kv_score_rescore adds to the word of the
 * kv_score_attention it follows.  The word keeps the first code posted to it
 * until the next such call or kv_check_status.
 *
 * Pointers: device pointers must be 16-byte aligned.  `stream` is a
 * cudaStream_t (NULL = legacy default stream).
 */
#ifndef KVEVICT_H
#define KVEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kv_status {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or shape */
    KV_ERR_BUDGET = 2,       /* a budget outside [sinks + w, n_r] */
    KV_ERR_WORKSPACE = 3,    /* workspace smaller than *_workspace_size */
    KV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    KV_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired */
    KV_ERR_UNSUPPORTED = 6   /* shape outside what the kernels handle */
} kv_status;

/* What kv_score sums over the window rows r that see key j (kv_problem.score_rule). */
typedef enum kv_score_rule {
    KV_SCORE_DROPKV = 0,          /* p_rj / (1 - p_rj) * ||a_r - v_j||_2 (DropKV)       */
    KV_SCORE_DROPKV_SQUARED = 1,  /* (p_rj / (1 - p_rj))^2 * ||a_r - v_j||_2^2          */
    KV_SCORE_ATTN_SUM = 2         /* p_rj (observation-window attention sum)            */
} kv_score_rule;

typedef struct kv_problem {
    int32_t num_requests;            /* R >= 0 (0: every call is a no-op) */
    int32_t num_layers;              /* L >= 1 */
    int32_t num_kv_heads;            /* H >= 1 */
    int32_t num_q_heads;             /* H_q, a multiple of H; G = H_q / H */
    int32_t head_dim;                /* d: 64 or 128 */
    int32_t window;                  /* w >= 1 */
    int32_t num_sinks;               /* s >= 0 (4 in the method) */
    int32_t score_rule;              /* kv_score_rule (0: the DropKV score) */
    const int64_t *seq_offsets_host; /* [R+1] cu_seqlens, host memory; n_r >= s + w, n_r < 2^31;
                                        L*H*N_tot and R*L*H_q*w below 2^31 (KV_ERR_UNSUPPORTED) */
    const int64_t *seq_offsets_dev;  /* the same [R+1] values, device memory */
    float softmax_scale;             /* logit scale, normally 1/sqrt(d); > 0 */
} kv_problem;

/* Bytes of workspace kv_score / kv_score_attention / kv_score_rescore need. */
kv_status kv_score_workspace_size(const kv_problem *p, size_t *bytes);

/*
 * Full scoring step: kv_score_attention then kv_score_rescore on one stream.
 * scores receives one fp32 score per key of every unit under p->score_rule,
 * >= 0 (the two DropKV rules give +inf when a window row puts all of its
 * attention on one key; the attention sum is at most G * w).  Results are
 * deterministic for a given problem.  The key-split size of the attention pass
 * is chosen from the whole problem's shape (enough work items for every SM), so
 * the same unit scored inside a problem of another shape may differ in the last
 * bits (within the stated tolerance of the exact score).
 */
kv_status kv_score(const kv_problem *p, const void *q_win, const void *k, const void *v,
                   float *scores, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Pass 1: causal window attention of every unit with split-K over the keys and
 * a merge of the splits (row max, row sum and a = sum p v); leaves them in the
 * workspace for pass 2.  Starts a new status sequence (zeroes the status word).
 * When the G*w window rows fit one 128-row chunk, p v multiplies bf16 v by p as
 * a bf16 hi/lo pair: V may take any finite bf16 value.  With more window rows it
 * runs with p and v in fp16: V values must then be below 65504 in magnitude
 * (bf16 values in that range convert exactly down to 2^-14 = 6.1e-5; smaller
 * magnitudes keep an absolute error below 3e-8).  A larger value posts
 * KV_ERR_UNSUPPORTED to the status word, and so does a block of 64 V rows as the
 * kernel reads them (64-aligned within the unit; the block at a unit's end also
 * holds the rows that follow it in memory) whose values are not all zero but all
 * below 2^-14 in magnitude, where fp16 keeps too few bits for the score's
 * tolerance (V scaled far below the usual range).  Rules that do not read V
 * (KV_SCORE_ATTN_SUM) have neither limit.
 */
kv_status kv_score_attention(const kv_problem *p, const void *q_win, const void *k,
                             const void *v, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Pass 2: rescoring of every key from the pass-1 results in the workspace.  Its
 * device status (a wait that expired) is added to the status word of the
 * kv_score_attention it follows; the word is not zeroed here. */
kv_status kv_score_rescore(const kv_problem *p, const void *q_win, const void *k,
                           const void *v, float *scores, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Max pooling of the scores, one unit at a time, over the keys outside the
 * observation window (the SnapKV convention the DropKV page follows: the w
 * window keys are kept anyway and are not pooled into their neighbours):
 *   scores_out[j] = max of scores_in[i], i in [j - r, j + r] within [0, n_r - w),
 *                   r = (kernel - 1) / 2, for j in [0, n_r - w);
 *   scores_out[j] = scores_in[j] for the window keys j in [n_r - w, n_r).
 * kernel: odd, 1..255 (11 on the DropKV page, 13 on the BellowsKV blog; 1
 * copies).  scores_in / scores_out: device f32 [L][H][N_tot], 16-byte
 * aligned, not overlapping (KV_ERR_INVALID_ARG otherwise).  The result feeds
 * kv_select_topk unchanged (pooled scores are still >= 0).
 */
kv_status kv_pool_scores(const kv_problem *p, int32_t kernel, const float *scores_in,
                         float *scores_out, void *stream);

/*
 * Host helper: offsets[u+1] = offsets[u] + budgets[u] for the R*L*H units,
 * offsets[0] = 0, after checking every budget lies in [s + w, n_r].
 * budgets_host [R*L*H] and offsets_host [R*L*H + 1] are host memory.
 */
kv_status kv_make_offsets(const kv_problem *p, const int32_t *budgets_host,
                          int64_t *offsets_host);

/* Bytes of workspace kv_select_topk and kv_head_budgets need. */
kv_status kv_select_workspace_size(const kv_problem *p, size_t *bytes);

/*
 * Per unit: keep the s sinks and the w window tokens, and from the middle
 * candidates [s, n_r - w) the budget - s - w highest scores, equal scores
 * going to the lower index.  Writes the kept indices, ascending, to
 * sel_idx[offsets[u] .. offsets[u+1]).  scores as written by kv_score (the
 * ordering compares the fp32 bit patterns, exact for values >= 0).
 * budgets_dev / offsets_dev: device copies of the tables above.  A budget
 * that is out of range, or disagrees with offsets, leaves its unit untouched
 * and posts KV_ERR_BUDGET to the select workspace's status word (zeroed at the
 * start of the call).
 */
kv_status kv_select_topk(const kv_problem *p, const float *scores, const int32_t *budgets_dev,
                         const int64_t *offsets_dev, int32_t *sel_idx, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Per-head budgets from the scores (DropKV page, Key Contributions "Adaptive
 * head budgets": DropKV scoring combined with AdaKV's head budget allocation).
 * For every (request, layer), the layer keeps as many tokens as budgets_dev
 * gives its H heads together; every head keeps its s sinks and w window
 * tokens, and the remaining slots go to the largest middle-candidate scores
 * [s, n_r - w) of all H heads together, equal scores to the lower head, then
 * the lower index.  budgets_out_dev[u] = s + w + the slots head u won;
 * offsets_out_dev = their exclusive scan (the per-layer totals, and so
 * offsets_dev[R*L*H], are unchanged).  Then kv_select_topk with the output
 * budgets keeps exactly the layer-wide winners, and kv_compact uses the output
 * offsets.
 * scores: as kv_score (or kv_pool_scores) writes them; budgets_dev, offsets_dev:
 * device [R*L*H] and [R*L*H + 1] as for kv_select_topk; outputs: device arrays
 * of the same sizes, distinct from the inputs.  workspace: at least
 * kv_select_workspace_size bytes (its status word is zeroed at the start of
 * the call; after the header, scratch).  A layer whose input budgets are out of
 * range or disagree with offsets_dev gets them copied through and posts
 * KV_ERR_BUDGET; the kv_select_topk that takes these outputs then fails the same
 * check on the same unit and posts KV_ERR_BUDGET again, so one kv_check_status
 * after the selection sees the error.
 * H * max n_r must be below 2^32 (KV_ERR_UNSUPPORTED otherwise).
 */
kv_status kv_head_budgets(const kv_problem *p, const float *scores, const int32_t *budgets_dev,
                          const int64_t *offsets_dev, int32_t *budgets_out_dev,
                          int64_t *offsets_out_dev, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * Block eviction (BellowsKV blog, eviction operator): one eviction decision
 * per block of `block_layers` consecutive layers, made from scores summed over
 * all layers and heads of the block, then applied to every layer and head of
 * the block.  The block view of a problem is the kv_problem with num_layers =
 * L / block_layers, num_kv_heads = num_q_heads = 1 and the same requests,
 * window and sinks; kv_pool_scores (13 in the blog), kv_budgets_fraction,
 * kv_make_offsets and kv_select_topk run on it unchanged.
 *
 * kv_block_scores: block_scores[b][t] = sum over the block's layers l (in
 * order) and heads h (in order) of scores[l][h][t], fp32, for every packed
 * token t.  scores: device f32 [L][H][N_tot]; block_scores: device f32
 * [L / block_layers][N_tot].  L must be a multiple of block_layers
 * (KV_ERR_INVALID_ARG otherwise).
 */
kv_status kv_block_scores(const kv_problem *p, int32_t block_layers, const float *scores,
                          float *block_scores, void *stream);

/*
 * Block form of kv_compact: unit u = (r, l, h) of p copies row i of its output
 * (offsets_dev[u] + i) from token block_sel_idx[block_offsets_dev[ub] + i],
 * ub = r * (L / block_layers) + l / block_layers, i.e. every layer and head of
 * a block keeps the tokens its block selected.  block_sel_idx /
 * block_offsets_dev: the selection and offsets of the block view;
 * offsets_dev: exclusive scan over p's units of the budgets, each unit's
 * budget being its block's.  Rows past the block's list, and out-of-range
 * indices, are skipped and left untouched.
 */
kv_status kv_compact_blocks(const kv_problem *p, int32_t block_layers, const void *k,
                            const void *v, const int32_t *block_sel_idx,
                            const int64_t *block_offsets_dev, const int64_t *offsets_dev,
                            int64_t total_rows, void *k_out, void *v_out, void *stream);

/*
 * k_out[offsets[u] + i] = k[row of unit u, token sel_idx[offsets[u] + i]],
 * the same for v: a bit copy of the kept rows into one packed ragged cache.
 * total_rows = offsets[R*L*H] (the caller knows it from kv_make_offsets).
 * Indices must be in [0, n_r); out-of-range ones are skipped and their output
 * rows left untouched.
 */
kv_status kv_compact(const kv_problem *p, const void *k, const void *v, const int32_t *sel_idx,
                     const int64_t *offsets_dev, int64_t total_rows, void *k_out, void *v_out,
                     void *stream);

/*
 * kv_score, kv_select_topk and kv_compact in ONE launch: the whole eviction
 * path (the score p/(1-p)*||a - v_j|| of DropKV, "Methodology in Plain English",
 * or the rule p->score_rule selects; the budgeted top-k with sinks and window
 * kept; the packed copy of the kept rows) as the phases of one persistent
 * cooperative kernel, one CTA per SM, separated by grid-wide barriers.  The
 * phases run the same device code as the three calls, so scores, sel_idx,
 * k_out and v_out are bit-identical to theirs.
 *
 * Arguments: those of kv_score (q_win, k, v, scores, workspace and its size:
 * the kv_score workspace), of kv_select_topk (budgets_dev, offsets_dev,
 * sel_idx) and of kv_compact (total_rows, k_out, v_out; with total_rows = 0
 * nothing is copied and k_out / v_out may be NULL).  Pooling and per-head
 * budgets are not part of the fused path: run kv_score, kv_pool_scores,
 * kv_head_budgets, kv_select_topk and kv_compact for those.
 *
 * Device-side errors go to the score workspace's status word
 * (kv_check_status): KV_ERR_BUDGET from the selection (that unit's indices are
 * not written), KV_ERR_UNSUPPORTED for V values fp16 cannot hold,
 * KV_ERR_TIMEOUT when a pipeline wait or a grid barrier wait exceeds the limit
 * of kv_set_wait_limit_ns (the kernel then skips its remaining phases and
 * returns).  KV_ERR_CUDA if the device cannot run a cooperative launch of one
 * CTA per SM.  Asynchronous on `stream` (an in-stream memset of the barrier
 * words precedes the kernel).
 */
kv_status kv_evict_fused(const kv_problem *p, const void *q_win, const void *k, const void *v,
                         const int32_t *budgets_dev, const int64_t *offsets_dev,
                         int64_t total_rows, float *scores, int32_t *sel_idx, void *k_out,
                         void *v_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The whole path for inputs and outputs in HOST memory (the end-to-end form of
 * kv_score + [kv_pool_scores] + [kv_head_budgets] + kv_select_topk +
 * kv_compact, or kv_evict_fused): the layers are processed in groups of
 * plan->group_layers; group g's window queries, K and V are copied to the
 * device on one internal stream while group g-1 is scored, selected and
 * compacted on `stream` and group g-2's kept indices and rows are copied back
 * on another, each copy one cudaMemcpyAsync.  The copies overlap the kernels
 * only when the host buffers are pinned (cudaHostAlloc / cudaHostRegister);
 * pageable buffers work, with the copies serialised.  Synchronous: returns
 * when the host outputs are complete.  The pages have no such entry point;
 * it exists so that a C caller can evict a cache that is not on the device.
 *
 * Inputs (host): q_win_host, k_host, v_host in the device layouts above;
 * budgets_host [R*L*H].  Outputs (host): offsets_host [R*L*H + 1] (the scan of
 * the budgets, or of the per-head budgets when plan->head_budgets is set),
 * sel_idx_host [offsets_host[R*L*H]], k_out_host / v_out_host
 * [offsets_host[R*L*H]][d] bf16 -- the standard unit order, bit-identical to
 * the device path on the same problem split into the same layer groups (each
 * group is scored as a problem of its own, so its pass-1 split size, chosen
 * from the group's shape, can differ from the whole problem's; scores then
 * differ in the last bits, within the score tolerance).
 * workspace: device memory of kv_evict_host_workspace_size bytes (two groups
 * of inputs, scores, workspaces and outputs, plus small tables), 16-byte
 * aligned.  Errors: as the calls it makes (KV_ERR_BUDGET from the host check of
 * the budgets before anything is copied); the device status of every group is
 * kept and the first nonzero code is returned in *device_status (KV_OK if
 * none).  Internal streams and events are created and destroyed per call.
 */
typedef struct kv_host_plan {
    int32_t group_layers;   /* layers per group, 1..L */
    int32_t pool_kernel;    /* 1 (no pooling) or an odd width up to 255 (kv_pool_scores) */
    int32_t head_budgets;   /* nonzero: per-head budgets (kv_head_budgets) within each layer */
    int32_t fused;          /* nonzero: kv_evict_fused per group (no pooling, no head budgets) */
} kv_host_plan;

kv_status kv_evict_host_workspace_size(const kv_problem *p, const kv_host_plan *plan,
                                       const int32_t *budgets_host, size_t *bytes);
kv_status kv_evict_host(const kv_problem *p, const kv_host_plan *plan, const void *q_win_host,
                        const void *k_host, const void *v_host, const int32_t *budgets_host,
                        int64_t *offsets_host, int32_t *sel_idx_host, void *k_out_host,
                        void *v_out_host, void *workspace, size_t workspace_bytes, void *stream,
                        int32_t *device_status);

/*
 * Synchronises `stream`, then reads and clears the device status word of a
 * score or select workspace.  *device_status receives the kv_status a kernel
 * posted (KV_OK if none).  Returns KV_ERR_CUDA if the stream itself reports an
 * error.  It takes the workspace because the library keeps no state between
 * calls: the word lives in the caller's workspace.
 */
kv_status kv_check_status(void *workspace, void *stream, int32_t *device_status);

/*
 * kv_score for callers that cannot allocate device memory.  No page these
 * kernels follow has a counterpart: it is a deployment convenience.
 *
 * Same inputs, outputs, layouts and asynchrony as kv_score, but the scratch
 * lives in one fixed 64 MiB array of device memory that belongs to this
 * library (held by every GPU that loads it, until the process exits), so the
 * caller passes no workspace.  It is meant for code that may not call the
 * CUDA allocator at run time -- a process that reserves all device memory at
 * start-up, a plugin whose host application owns the allocator, a path that
 * must avoid cudaMalloc's implicit synchronisation.  It allocates nothing.
 *
 *  - Problems whose kv_score workspace (kv_score_workspace_size) exceeds
 *    64 MiB return KV_ERR_WORKSPACE before anything is launched.
 *  - The first call in each CUDA context (per device, and again after
 *    cudaDeviceReset or when another context is made current) looks up the
 *    array's device address with that context current, and later calls in
 *    the same context reuse it (keyed on the context's unique ID); make the
 *    first call of a context before any stream capture.
 *  - Every call shares the array and it keeps the last call's contents;
 *    calls that overlap on the GPU (other streams or host threads on the same
 *    device) race on it, so order them on one stream.
 *  - Argument and launch errors are returned.  The device-side status that
 *    kv_score posts to its workspace (kv_check_status) lands in the shared
 *    array and is not reported here: a wait that expired (KV_ERR_TIMEOUT) and,
 *    with more than 128 window rows, V values outside what pass 1 carries in
 *    fp16 (KV_ERR_UNSUPPORTED: |v| of 65504 or more, or 64-row blocks of values
 *    all below 2^-14; see kv_score_attention) then leave wrong scores without
 *    an error.  Callers whose V may leave that range should use kv_score with a
 *    workspace.
 */
kv_status kv_score_noalloc(const kv_problem *p, const void *q_win, const void *k,
                           const void *v, float *scores, void *stream);

/*
 * Watchdog of the device waits.  Every wait inside the tensor-core kernels (a
 * pipeline stage, a tensor-core result) gives up after `ns` nanoseconds,
 * posts KV_ERR_TIMEOUT to the workspace status word (read it with
 * kv_check_status) and lets the kernel return with the context usable; the
 * kernel's waits for its own copies and MMAs still in flight always allow
 * 2 s.  Process-wide; applies to launches made after the call.  The default
 * is 2e9 (2 s); 0 makes every wait that is not already satisfied give up at
 * once, which exercises the failure path.  No page has a counterpart: this
 * is the library's own failure detection.
 */
void kv_set_wait_limit_ns(uint64_t ns);
uint64_t kv_get_wait_limit_ns(void);

/* Static, human-readable name of a status code. */
const char *kv_status_string(kv_status s);

/*
 * Host helpers: per-layer budgets b_l (tokens per KV head) whose sum is
 * exactly L*B.  Real targets B*m_l are rounded by largest remainder: floor
 * each, then one more token to the layers with the largest fractional parts,
 * ties to the lower layer.
 *   pyramid: m_l proportional to lo + (hi - lo) * (1 - l/(L-1))^curve, mean 1
 *            (PyramidKV guide; hi = 1.8, lo = 0.2, curve = 1 is linear).
 *   ripple:  s_hat = min-max normalised profile (all 0 if constant), m_l
 *            proportional to exp(beta * s_hat_l) clipped to [1/gamma, gamma]
 *            (gamma = +inf: no clip), then mean 1 (RippleKV Eq. (9)-(11)).
 * budgets_out: host [L].
 */
kv_status kv_budgets_pyramid(int32_t num_layers, int32_t mean_budget, double hi, double lo,
                             double curve, int32_t *budgets_out);
kv_status kv_budgets_ripple(int32_t num_layers, int32_t mean_budget, const double *profile,
                            double beta, double gamma, int32_t *budgets_out);

/*
 * Host helper: budgets_host[u] = s + w + floor(q * (n_r - s - w)) for every
 * unit of p: the sinks and window kept and the fraction q (in [0, 1]) of the
 * rest (BellowsKV blog, eviction operator: the fraction q of the remaining
 * positions survives).  budgets_host: host [R*L*H].
 */
kv_status kv_budgets_fraction(const kv_problem *p, double q, int32_t *budgets_host);

#ifdef __cplusplus
}
#endif

#endif /* KVEVICT_H */
