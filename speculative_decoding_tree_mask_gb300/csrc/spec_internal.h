// Host-side launch interface between the C ABI (api.cu) and the kernels. Internal.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace specv {

// Launches `kernel` on `st` allowing it to start before the previous kernel in the stream has
// finished (programmatic dependent launch): the kernel must call grid_dep_wait() before it
// reads anything an earlier kernel writes. Hides the launch latency between the stages.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The same for a kernel launched in thread-block clusters of `cluster` CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_dependent_cluster(void (*kernel)(Params...), dim3 grid, dim3 block,
                                     size_t smem, cudaStream_t st, int cluster,
                                     Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

constexpr int kMaxN = 64;   // nodes per request (one 64-bit ancestor mask)

// Shapes of the row-statistics stream. The one-CTA-per-row kernel keeps SPEC_ROW_MIN_CTAS
// CTAs of 256 threads on every SM with SPEC_ROW_UNROLL 16-byte loads in flight per thread;
// the split kernel (small batches: several CTAs per row, one wave) has its own pair, since
// with fewer CTAs than the GPU can hold it can trade occupancy for bytes in flight.
#ifndef SPEC_ROW_UNROLL
#define SPEC_ROW_UNROLL 4
#endif
#ifndef SPEC_ROW_MIN_CTAS
#define SPEC_ROW_MIN_CTAS 6
#endif
#ifndef SPEC_SPLIT_UNROLL
#define SPEC_SPLIT_UNROLL 4
#endif
#ifndef SPEC_SPLIT_MIN_CTAS
#define SPEC_SPLIT_MIN_CTAS 6
#endif
// The paired target + dense-draft launch likewise: its dense-draft rows keep more values live,
// which at 6 CTAs per SM (40 registers) spilled; 5 per SM fit without spills.
#ifndef SPEC_PAIR_UNROLL
#define SPEC_PAIR_UNROLL 4
#endif
#ifndef SPEC_PAIR_MIN_CTAS
#define SPEC_PAIR_MIN_CTAS 5
#endif
constexpr int kRowCtasPerSm = SPEC_ROW_MIN_CTAS;
constexpr int kSplitCtasPerSm = SPEC_SPLIT_MIN_CTAS;

enum RowMode { ROW_GREEDY = 0, ROW_SAMPLE = 1, ROW_PROBS = 2 };

// Row chunks: the row-statistics stream splits every row into kRowChunks contiguous pieces
// and, for sampling rows that start 16-byte aligned, stores each piece's (max, sum) so that
// the inverse-CDF bonus re-reads one piece instead of the row.
#ifndef SPEC_ROW_CHUNKS
#define SPEC_ROW_CHUNKS 8
#endif
constexpr int kRowChunks = SPEC_ROW_CHUNKS;
static_assert(kRowChunks == 1 || kRowChunks == 2 || kRowChunks == 4 || kRowChunks == 8,
              "row chunks: a power of two that divides the 8 warps of the stream");
constexpr int kSubTile = 256;   // elements per sub-tile of the walk's bonus search

// The lazy walks split the rows they stream into one chunk per warp of their 512 threads.
constexpr int kLazyChunks = 16;

// First vector of chunk c (c = 0..nc) of a row of nv 16-byte vectors holding epv elements
// each, for a split into nc chunks. Aligned rows cut on sub-tile boundaries (as balanced as
// whole sub-tiles allow), so chunk c covers elements
// [row_chunk_sub(c) * kSubTile, row_chunk_sub(c + 1) * kSubTile) clipped to V; other rows
// split the vectors evenly.
__host__ __device__ __forceinline__ int row_chunk_sub(int c, int64_t V, int nc = kRowChunks) {
    const int64_t nsub = (V + kSubTile - 1) / kSubTile;
    return (int)(nsub * c / nc);
}
__host__ __device__ __forceinline__ int row_chunk_vec(int c, int nv, int64_t V, bool aligned,
                                                      int epv, int nc = kRowChunks) {
    if (c >= nc) return nv;
    if (!aligned) return (int)((int64_t)nv * c / nc);
    const int64_t v = (int64_t)row_chunk_sub(c, V, nc) * (kSubTile / epv);
    return v < nv ? (int)v : nv;
}
enum DraftKind { DRAFT_POINT = 0, DRAFT_PROBS_F32 = 1, DRAFT_LOGITS = 2 };

// Partial statistics of a piece of a row: max, sum of 2^((x - max) k), lowest index of the
// max, flags.
struct RowPart {
    float m, s;
    int arg, flags;
};

// Row statistics over `rows` rows of V elements (see spec_row_stats in spec_verify.h).
struct RowStatsParams {
    const void *x;
    int64_t V;
    int rows;
    int N;                   // nodes per request; rows are (b, n) = (row / N, row % N)
    float k;                 // log2(e) / T (sampling); unused for greedy / probabilities
    const int32_t *parent;   // with tok: gather of child probabilities; may be null
    const int32_t *tok;
    int skip_leaves;         // rows of nodes without children are not read (draft rows)
    float *m;
    float *s;
    int32_t *arg;
    int32_t *flags;
    float *pc;               // child_prob output (indexed by child row); may be null
    int pc_normalized;       // 1: pc = e_t / S (probability); 0: pc = e_t (walk input)
    const int32_t *n_active = nullptr;   // per-request node budget [B]; null = all N rows
    float2 *chunk = nullptr;   // sampling: (max, sum) of each row chunk [rows, kRowChunks]
    // Small batches: with piece and count set and split in {2, 4, 8}, each row is streamed by
    // `split` CTAs; piece holds their partial statistics [rows, split], count their arrivals
    // [rows] (zero between launches).
    RowPart *piece = nullptr;
    int32_t *count = nullptr;
    int split = 1;
    int32_t *dbg = nullptr;   // debug builds: per-request violation bits [B] (may be null)
};

cudaError_t launch_row_stats(const RowStatsParams &p, int dtype, int mode, cudaStream_t st);
// Sampling statistics of the target rows and of the dense-draft rows in one launch.
cudaError_t launch_row_stats_pair(const RowStatsParams &target, int dtype,
                                  const RowStatsParams &draft, int draft_dtype, int draft_mode,
                                  cudaStream_t st);

cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                             int32_t *status, cudaStream_t st);

struct WalkOutputs {
    int32_t *accept_len;
    int32_t *out_tokens;
    int32_t *kv_commit;
    int32_t *bonus;
    int32_t *status;
};

struct GreedyWalkParams {
    int B, N;
    int64_t V;
    const int32_t *parent, *tok;
    const int32_t *arg, *flags;   // row statistics [B, N]
    WalkOutputs out;
    const int32_t *n_active = nullptr;
    int32_t *dbg = nullptr;       // debug builds: per-request violation bits [B]
};

cudaError_t launch_walk_greedy(const GreedyWalkParams &p, cudaStream_t st);

// Greedy verification reading only the rows on the accepted path (one CTA per request).
struct LazyGreedyParams {
    int B, N;
    int64_t V;
    int dtype;
    const void *logits;
    const int32_t *parent, *tok;
    WalkOutputs out;
    const int32_t *n_active = nullptr;
    int32_t *dbg = nullptr;       // debug builds: per-request violation bits [B]
};

cudaError_t launch_lazy_greedy(const LazyGreedyParams &p, cudaStream_t st);

struct SampleWalkParams {
    int B, N;
    int64_t V;
    int dtype;                    // target logits element type
    const void *logits;
    const int32_t *parent, *tok;
    const float *uniforms;        // [B, N+1]
    float k;                      // log2(e) / T
    // target row statistics [B, N] and child probabilities p_parent(tok[c]) [B, N]
    const float *m, *s, *pc;
    const int32_t *flags;
    // dense draft (kind != DRAFT_POINT)
    int draft_kind, draft_dtype;
    const void *draft;
    const float *mq, *sq, *qc;
    const int32_t *dflags;
    int lazy;                     // 1: no row statistics precomputed; stream visited rows only
    int host_rows = 0;            // lazy: the logits are in host memory (read over the link)
    WalkOutputs out;
    const int32_t *n_active = nullptr;
    const float2 *chunk = nullptr;   // row-chunk partials of the target rows (eager, may be null)
    // Eager walks: CTAs per request (1, 2, 4 or 8), one thread-block cluster each; the
    // cluster splits every vocabulary pass of its request.
    int cluster = 1;
    int32_t *dbg = nullptr;       // debug builds: per-request violation bits [B]
};

// KV commit of the accepted path into a paged cache (see spec_kv_commit).
struct KvCommitParams {
    const void *src_k, *src_v;
    int src_dtype;                // 0 f32, 1 bf16, 2 f16
    int B, N, H, D;
    const int32_t *kv_commit, *accept_len;
    void *cache_k, *cache_v;
    int cache_kind;               // 0 source type, 1 fp8 e4m3, 2 fp8 e5m2
    int layout;                   // 0 NHD, 1 HND
    int block_size;
    int64_t num_blocks;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *seq_pos;
    const float *k_scale, *v_scale;
    int scale_per_token;          // 1: scales are [B, N], per source token
    int32_t *status;
    int sms;                      // SMs of the device (the grid is a few CTAs per SM)
};

cudaError_t launch_kv_commit(const KvCommitParams &p, bool vec, cudaStream_t st);

// Adaptive node-budget update (see spec_budget_update).
struct BudgetParams {
    spec_budget_params prm;
    const int32_t *accept_len, *status, *parent;
    int B, N;
    spec_budget_state *state;
    int32_t *n_active;
};

cudaError_t launch_budget_update(const BudgetParams &p, cudaStream_t st);

cudaError_t launch_walk_sample(const SampleWalkParams &p, cudaStream_t st);

}  // namespace specv
