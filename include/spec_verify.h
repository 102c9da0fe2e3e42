/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding verification library.
 *
 * The operation (EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless
 * throughput", commit 4b728e2 "grammar-trie tree speculation with exact acceptance"): the
 * draft is a trie of N nodes (node 0 is the root, the last committed token) whose logits the
 * target model produced in one tree-attention forward, one row per node. Verification turns
 * those rows into an exact accept/reject decision per request: greedy decoding keeps the
 * argmax path, sampling uses standard (SpecInfer-style) rejection sampling against the draft
 * so the output distribution equals the target's, and a bonus token is drawn where the walk
 * stops. IluvatarLabs/vllm PR #3 "SCV vectorized masking" computes the per-request
 * acceptance mask on the device without host synchronisation; this library likewise never
 * synchronises with the host inside a call.
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers owned by the caller, row-major and contiguous.
 *     They must be aligned to their element size. Logits rows have stride V elements.
 *   - Tree: parent int32 [B, N] with parent[b][0] == -1 and 0 <= parent[b][i] < i
 *     (topological order); draft_token int32 [B, N], entry 0 (the root) is ignored. Children
 *     of a node are visited in ascending node index ("trie order"). 1 <= N <= 64.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream) and
 *     never synchronise the host. One handle serves one stream at a time (its workspace is
 *     reused by every call).
 *   - Host-checkable problems (NULL handle or pointer, sizes beyond the handle's limits,
 *     unknown dtype, bad temperature) return a negative SPEC_ERR_* code synchronously and
 *     launch nothing. Problems in the data are reported per request in status[b]
 *     (SPEC_REQ_*); a request with nonzero status gets accept_len 0, bonus -1 and -1 in
 *     every out_tokens / kv_commit slot. SPEC_ERR_CUDA means a launch failed.
 *   - Outputs of a verify call, per request b:
 *       accept_len[b]          number of accepted non-root nodes L;
 *       out_tokens[b][0..L]    draft tokens of the accepted nodes in path order, then the
 *                              bonus token; -1 beyond L;
 *       kv_commit[b][0..L]     node ids whose KV entries to keep: 0 (the root, produced by
 *                              the same forward) then the accepted nodes; -1 beyond L;
 *       bonus[b]               the bonus token;  status[b]  SPEC_REQ_*.
 *     out_tokens and kv_commit are int32 [B, N].
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_ctx *spec_handle;

enum {
    SPEC_OK = 0,
    SPEC_ERR_ARG = -1,          /* an argument is invalid or outside the handle's limits */
    SPEC_ERR_UNSUPPORTED = -2,  /* a valid request the library does not implement */
    SPEC_ERR_CUDA = -3,         /* a CUDA call or launch failed */
    SPEC_ERR_WORKSPACE = -4     /* workspace allocation failed */
};

enum { SPEC_F32 = 0, SPEC_BF16 = 1, SPEC_F16 = 2 };  /* element types (F16: K/V only) */

enum {
    SPEC_DRAFT_POINT = 0,       /* deterministic trie: the draft puts mass 1 on each child */
    SPEC_DRAFT_PROBS_F32 = 1,   /* draft probabilities float32 [B, N, V], used as given */
    SPEC_DRAFT_LOGITS = 2       /* draft logits [B, N, V] (SPEC_F32 / SPEC_BF16), softmax(d/T) */
};

enum {
    SPEC_REQ_OK = 0,
    SPEC_REQ_BAD_PARENT = 1,    /* parent[0] != -1 or parent[i] outside [0, i) */
    SPEC_REQ_BAD_TOKEN = 2,     /* a non-root draft token outside [0, V) */
    SPEC_REQ_BAD_ROW = 3,       /* a row the walk needs holds NaN / +inf or is all -inf
                                   (for probabilities: NaN, inf or a negative entry) */
    SPEC_REQ_BAD_UNIFORM = 4,   /* a uniform in slots 1..N is NaN or outside [0, 1) */
    SPEC_REQ_BAD_SLOT = 5,      /* KV commit: a slot maps outside the block table or cache */
    SPEC_REQ_BAD_BUDGET = 6,    /* the request's node budget (spec_set_node_budget) is
                                   outside [1, N] */
    SPEC_REQ_INTERNAL = 7       /* debug builds only (SPEC_DEBUG): one of the kernels' own
                                   consistency checks failed for this request -- an index
                                   outside its array (the access was skipped), a split row's
                                   arrival counter outside [0, split), or an accepted path that
                                   is not a chain of parent links; see spec_debug_words */
};

enum { SPEC_KV_NHD = 0, SPEC_KV_HND = 1 };  /* paged KV cache layouts */
enum { SPEC_CACHE_SAME = 0, SPEC_CACHE_FP8_E4M3 = 1, SPEC_CACHE_FP8_E5M2 = 2 };
enum { SPEC_SCALE_TENSOR = 0, SPEC_SCALE_PER_TOKEN = 1 };   /* fp8 KV scale forms */

/* Row-statistics flag bits (spec_row_stats row_flags). */
enum { SPEC_ROW_NAN = 1, SPEC_ROW_POSINF = 2, SPEC_ROW_ALL_NEGINF = 4 };

/* Kernel classes reported by the profiling calls. */
enum {
    SPEC_K_TREE_MASK = 0,
    SPEC_K_ROW_STATS = 1,       /* target logits rows */
    SPEC_K_DRAFT_STATS = 2,     /* reserved: dense draft rows now share the ROW_STATS launch */
    SPEC_K_WALK_GREEDY = 3,
    SPEC_K_WALK_SAMPLE = 4,
    SPEC_K_LAZY_GREEDY = 5,
    SPEC_K_LAZY_SAMPLE = 6,
    SPEC_K_KV_COMMIT = 7,
    SPEC_K_BUDGET = 8,          /* adaptive node-budget update */
    SPEC_K_COUNT = 9
};

/*
 * Create a handle for `device` able to serve calls with B <= max_B, N <= max_N (<= 64) and
 * V <= max_V (<= 2^21). Allocates a device workspace of 232 * max_B * max_N + 4 * max_B
 * bytes with cudaMalloc (released by spec_verify_destroy). Returns SPEC_ERR_ARG for out-of-range limits,
 * SPEC_ERR_CUDA if the device cannot be used, SPEC_ERR_WORKSPACE if allocation fails.
 */
int spec_verify_init(spec_handle *h, int max_B, int max_N, int64_t max_V, int device);

/* Free the handle and its workspace. Waits for nothing: the caller must ensure no call on
 * the handle is still running. NULL is accepted. */
int spec_verify_destroy(spec_handle h);

/*
 * Tree-attention mask (EmbodiInfer PR #11, commit 4b728e2: all N nodes are verified in one
 * tree-attention forward; IluvatarLabs/vllm PR #3: the mask is built on the device).
 * anc_mask uint64 [B, N]: bit j of anc_mask[b][i] is set iff node j is node i or one of its
 * ancestors, i.e. query i may attend to key j. depth int32 [B, N]: number of edges from the
 * root. status int32 [B]: SPEC_REQ_OK or SPEC_REQ_BAD_PARENT (then the request's masks are 0
 * and depths -1).
 */
int spec_build_tree_mask(spec_handle h, const int32_t *parent, int B, int N, uint64_t *anc_mask,
                         int32_t *depth, int32_t *status, void *stream);

/*
 * Greedy verification (EmbodiInfer PR #11, commit 4b728e2: greedy keeps the argmax path).
 * logits [B, N, V] of `dtype` (SPEC_F32 / SPEC_BF16). From the root, repeatedly take
 * a = argmax of the current node's row (lowest index on ties) and move to the first child in
 * trie order whose draft token equals a; stop when none does. The bonus is a at the stop
 * node. Rows of nodes off the path never influence an output (NaN there is harmless).
 */
int spec_verify_greedy(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                       const int32_t *draft_token, const int32_t *parent, int32_t *accept_len,
                       int32_t *out_tokens, int32_t *kv_commit, int32_t *bonus, int32_t *status,
                       void *stream);

/*
 * Sampling verification (EmbodiInfer PR #11, commit 4b728e2: standard rejection sampling
 * against the draft, output distribution unchanged). p = softmax(z / temperature) per row;
 * temperature == 0 runs spec_verify_greedy (the draft and uniforms are then ignored);
 * temperature must be finite and >= 0.
 * uniforms float32 [B, N+1] in [0, 1): slot c is consumed when child c is tested, slot N
 * draws the bonus, slot 0 is unused.
 *   SPEC_DRAFT_POINT (draft NULL): at a node with rejected-token set R, child c with token t
 *     is accepted iff u[c] < p(t) / sum_{v not in R} p(v) (0 if t is in R); on rejection t
 *     joins R; when the walk stops the bonus is the inverse CDF of p with R zeroed at u[N].
 *   SPEC_DRAFT_PROBS_F32 / SPEC_DRAFT_LOGITS: draft row i is the distribution q that drafted
 *     node i's children (the same temperature is applied to draft logits). Child c with
 *     token x is accepted iff u[c] * q(x) < r(x), r starting as p; on rejection
 *     r <- max(r - q, 0) / sum(max(r - q, 0)) (kept unchanged if that sum is 0); the bonus is
 *     the inverse CDF of r at u[N] (of p at a leaf). On a chain this is standard speculative
 *     sampling; on a tree, siblings are taken as independent draws from q.
 * Inverse CDF: with S = sum r and tau = u*S, the smallest v whose running sum exceeds tau
 * (the largest v with r(v) > 0 if rounding leaves none).
 */
int spec_verify_sample(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                       const int32_t *draft_token, const int32_t *parent, const void *draft,
                       int draft_kind, int draft_dtype, float temperature,
                       const float *uniforms, int32_t *accept_len, int32_t *out_tokens,
                       int32_t *kv_commit, int32_t *bonus, int32_t *status, void *stream);

/*
 * Lazy verification: the same operations, arguments, results and status codes as
 * spec_verify_greedy / spec_verify_sample, but only the rows the walk visits are read (the
 * accepted path and the stop node: at most depth + 1 rows per request, plus, for dense
 * drafts, the draft rows of the visited inner nodes), one CTA per request, instead of a
 * first pass over all B*N rows. EmbodiInfer PR #11 (commit 4b728e2) verifies all trie nodes
 * in one forward; the walk decides on few of them, so the rows of nodes off the path never
 * need to be read. Greedy results are bit-identical to the eager call; sampling results can
 * differ from it only where float32 rounding of a sum decides (the same margin cases as
 * against the float64 reference). Rows are streamed one after another along the path, so the
 * latency grows with the accepted length.
 * Here (only) logits and draft may also be page-locked host memory that the device maps at
 * the same address (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped on a
 * system with unified addressing): the visited rows are then read directly over the host
 * link, with no copy of the other rows. Other host memory, and device memory of a GPU other
 * than the handle's, return SPEC_ERR_ARG (checked with cudaPointerGetAttributes).
 */
int spec_verify_greedy_lazy(spec_handle h, const void *logits, int dtype, int B, int N,
                            int64_t V, const int32_t *draft_token, const int32_t *parent,
                            int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                            int32_t *bonus, int32_t *status, void *stream);
int spec_verify_sample_lazy(spec_handle h, const void *logits, int dtype, int B, int N,
                            int64_t V, const int32_t *draft_token, const int32_t *parent,
                            const void *draft, int draft_kind, int draft_dtype, float temperature,
                            const float *uniforms, int32_t *accept_len, int32_t *out_tokens,
                            int32_t *kv_commit, int32_t *bonus, int32_t *status, void *stream);

/*
 * KV commit after verification (IluvatarLabs/vllm PR #3, commit_draft_kernel: the K/V of
 * accepted draft tokens are copied into the paged cache, NHD or HND, fp16/bf16/fp32 sources,
 * a cache of the source type or fp8 with a scale, rejected entries skipped; EmbodiInfer PR #11,
 * commits 938fe7b and 41dcd00: only the new tokens are committed).
 *   src_k, src_v    [B, N, H, D] of src_dtype (SPEC_F32 / SPEC_BF16 / SPEC_F16): the K/V the
 *                   verify forward produced for every tree node;
 *   kv_commit, accept_len   outputs of a verify call ([B, N] and [B]);
 *   cache_k, cache_v        paged caches, layout SPEC_KV_NHD [num_blocks, block_size, H, D] or
 *                   SPEC_KV_HND [num_blocks, H, block_size, D]; element type: the source type
 *                   (SPEC_CACHE_SAME) or one byte of fp8 (SPEC_CACHE_FP8_E4M3 / _E5M2);
 *   block_table     int32 [B, max_blocks]: cache block of each block_size tokens of request b;
 *   seq_pos         int32 [B]: sequence position of slot 0 (the root);
 *   k_scale, v_scale        device float32 scales for fp8 caches (NULL = 1): the cache stores
 *                   the fp8 rounding (nearest, ties to even, saturated) of x / scale;
 *   scale_per_token SPEC_SCALE_TENSOR: each scale is one value; SPEC_SCALE_PER_TOKEN: each is
 *                   float32 [B, N], the scale of source token (b, node) (the commit kernel of
 *                   IluvatarLabs/vllm PR #3 takes scalar and per-token scales);
 *   commit_status   int32 [B] (may be NULL): SPEC_REQ_BAD_SLOT if a slot's position or block
 *                   falls outside the table or the cache (that slot is skipped), else 0.
 * Slot j of request b (j = 0..accept_len[b]) is written at position seq_pos[b] + j. Requests
 * whose kv_commit[b][0] is negative (verification failed) write nothing.
 */
int spec_kv_commit(spec_handle h, const void *src_k, const void *src_v, int src_dtype, int B,
                   int N, int H, int D, const int32_t *kv_commit, const int32_t *accept_len,
                   void *cache_k, void *cache_v, int cache_kind, int layout, int block_size,
                   int64_t num_blocks, const int32_t *block_table, int max_blocks,
                   const int32_t *seq_pos, const float *k_scale, const float *v_scale,
                   int scale_per_token, int32_t *commit_status, void *stream);

/*
 * The vocabulary-streaming row statistics on their own (the first stage of both verify
 * calls), for `rows` contiguous rows of V elements:
 *   row_max[r]    max_v z[r][v] (float32; exact for bf16/f32 inputs)
 *   row_argmax[r] lowest index attaining it
 *   row_sum[r]    sum_v exp((z[r][v] - row_max[r]) / temperature), or 0 when temperature == 0
 *   row_flags[r]  SPEC_ROW_* bits (nonzero = the row is unusable for verification)
 * If draft_token, parent and child_prob are all non-NULL the rows are read as [B, N, V]
 * with B = rows / N, and child_prob[b][c] = p_{parent(c)}(draft_token[b][c]) for every
 * non-root node c whose parent is in range and whose token is in [0, V) (other slots are
 * left untouched); temperature must then be > 0.
 */
int spec_row_stats(spec_handle h, const void *logits, int dtype, int rows, int N, int64_t V,
                   float temperature, const int32_t *draft_token, const int32_t *parent,
                   float *row_max, float *row_sum, int32_t *row_argmax, int32_t *row_flags,
                   float *child_prob, void *stream);

/*
 * Per-kernel timing. After spec_profile_begin, every kernel launched through the handle is
 * bracketed with CUDA events on its stream (at most 16384 launches are recorded).
 * spec_profile_end waits for those events and writes, per SPEC_K_* class, the summed
 * device milliseconds and the number of launches, then stops recording.
 */
int spec_profile_begin(spec_handle h);
int spec_profile_end(spec_handle h, float *ms_per_class, int32_t *launches_per_class);

/*
 * Node budget (IluvatarLabs/vllm PR #3, adaptive mode: the number of speculative tokens
 * verified per step follows the recent acceptance ratio, and the mask computation is replayed
 * from captured CUDA graphs). Draft nodes are in topological order, so the first n nodes of a
 * tree always form a tree themselves; a budget of n keeps exactly those.
 *
 * spec_set_node_budget makes every later verify call on the handle (eager and lazy, greedy
 * and sampling) read n_active[b] -- a DEVICE int32 [>= B] array owned by the caller, read by
 * the kernels when they run -- and verify request b as the tree of its nodes 0..n-1 with
 * n = n_active[b]: nodes >= n do not exist for that call (their rows are not read, their
 * tokens, parents and uniform slots are not checked), while shapes, the bonus uniform slot N
 * and the [B, N] output layout stay as they are. A value outside [1, N] gives that request
 * SPEC_REQ_BAD_BUDGET. Because the value is read on the device, a CUDA graph captured once
 * follows every new budget on replay. NULL (the default) verifies all N nodes. The array must
 * stay valid while it is set. spec_row_stats and spec_verify_greedy_noalloc ignore it.
 */
int spec_set_node_budget(spec_handle h, const int32_t *n_active);

/*
 * Budget controller, one update per verify step, entirely on the device (no host
 * synchronisation, so it can sit inside a captured graph next to the verify call).
 *   params (host struct, copied at the call):
 *     target   acceptance ratio to hold, in (0, 1];
 *     alpha    weight of the newest step in the moving average, in (0, 1];
 *     band     dead band around the target, finite and >= 0;
 *     n_min, n_max   budget limits, 1 <= n_min <= n_max <= N;  step   change per update, >= 1.
 *   accept_len, status  int32 [B]: outputs of the verify call the budget governed;
 *   parent      int32 [B, N]: that call's trees;
 *   state       DEVICE spec_budget_state, caller-owned and initialised by the caller (ema,
 *               budget; steps = 0), read and rewritten by the update;
 *   n_active    DEVICE int32 [B]: on entry the budgets the verify call used; on exit every
 *               entry holds the new budget.
 * Update: over requests with status 0 and a budget n in [1, N], A = sum of accept_len and
 * D = sum of the deepest node depth among nodes 0..n-1 (the most that request could have
 * accepted). If D > 0: ratio = A / D, ema <- (1 - alpha) * ema + alpha * ratio, steps += 1;
 * the budget (first clamped to [n_min, n_max]) rises by step (at most n_max) when
 * ema > target + band and falls by step (at least n_min) when ema < target - band. If D == 0
 * the average is unchanged. All of it is evaluated in float64 in this order, so the result is
 * reproducible exactly. Bad parameters return SPEC_ERR_ARG and launch nothing.
 */
typedef struct {
    double target, alpha, band;
    int32_t n_min, n_max, step;
} spec_budget_params;

typedef struct {
    double ema;       /* moving average of the acceptance ratio */
    int32_t budget;   /* node budget for the next step */
    int32_t steps;    /* updates that saw at least one usable request */
} spec_budget_state;

int spec_budget_update(spec_handle h, const spec_budget_params *params,
                       const int32_t *accept_len, const int32_t *status, const int32_t *parent,
                       int B, int N, spec_budget_state *state, int32_t *n_active, void *stream);

/* Static description of a SPEC_ERR_* code. */
const char *spec_error_string(int code);

/*
 * Debug flavour. The library built with SPEC_DEBUG (libspecverify_debug.so) runs the same
 * kernels with their own consistency checks compiled in: every vector index of the vocabulary
 * streams, every store into the walks' shared arrays, the accepted path (a chain of parent
 * links from the root), the bonus token (in [0, V), not a rejected token), the KV commit's
 * source and cache indices, and the split rows' arrival counters (each arrival must see a
 * value in [0, split)). A failed check skips the access, sets a bit in the request's debug
 * word (1 index, 2 arrival counter, 4 walk) and turns the request's result into
 * SPEC_REQ_INTERNAL (the KV commit's status likewise). Nothing traps or waits. Each verify
 * call of the debug build first zeroes the debug words of its requests and all arrival
 * counters. The EmbodiInfer PR #11 commit e9133f4 lesson (stale NaN slots must not reach an
 * output) and the TensorRT-LLM PR #16953 debug-flagged checks motivate this flavour.
 *
 * spec_debug_build: 1 in the debug build, 0 otherwise.
 * spec_debug_inject_arrival: arms a one-shot fault injection for tests: the next verify call
 *   on the handle whose row statistics are split over several CTAs per row writes `value`
 *   into the arrival counter of row `row` (b * N + node) after zeroing the counters, so its
 *   check must catch it. Returns SPEC_ERR_UNSUPPORTED in release builds.
 * spec_debug_words: copies the debug words of requests 0..B-1 of the handle's last call into
 *   the device int32 array `words` (asynchronously on `stream`). SPEC_ERR_UNSUPPORTED in
 *   release builds.
 */
int spec_debug_build(void);
int spec_debug_inject_arrival(spec_handle h, int row, int value);
int spec_debug_words(spec_handle h, int32_t *words, int B, void *stream);

/*
 * Greedy verification that allocates nothing. The pages have no counterpart of this entry
 * point; it exists for callers that cannot call cudaMalloc, for example plugins inside an
 * engine that reserves all device memory up front and hands a kernel only its tensors, or
 * latency-critical loops that cannot accept cudaMalloc's implicit device synchronisation.
 *
 * Same arguments, results and status codes as spec_verify_greedy, but no handle: it runs on
 * the current device, and the per-row scratch (argmax and flags of each of the B*N rows) is
 * a static device array of SPEC_NOALLOC_MAX_ROWS rows (128 KiB) that every GPU loading the
 * library holds until the process exits. B*N > SPEC_NOALLOC_MAX_ROWS returns SPEC_ERR_ARG
 * and launches nothing, and so do logits that are not memory of the current device
 * (checked with cudaPointerGetAttributes). No cudaMalloc, cudaFree or allocating library
 * call is made.
 * The first call in a CUDA context looks up the array's device address in that context
 * (cudaGetSymbolAddress) and caches it with the context's ID; make that first call before
 * any stream capture. A new context on the device (after cudaDeviceReset, or another
 * driver-API context made current) loads the library's module at a new address: the next
 * call sees the new context ID and looks the address up again, so it too should come before
 * any capture. All calls share the one array (each call writes every row it reads, so stale
 * contents do not matter), so calls that overlap on the GPU, on any streams, race:
 * serialise them.
 */
#define SPEC_NOALLOC_MAX_ROWS 16384
int spec_verify_greedy_noalloc(const void *logits, int dtype, int B, int N, int64_t V,
                               const int32_t *draft_token, const int32_t *parent,
                               int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                               int32_t *bonus, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
