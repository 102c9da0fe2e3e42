// Vocabulary-streaming row statistics: one CTA per (request, node) row.
//
// EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput"
// (commit 4b728e2) verifies the N trie nodes in one forward, so every node has a logits row;
// acceptance needs, per row, the argmax (greedy), and the softmax normaliser at temperature T
// plus p at the drafted child tokens (rejection sampling). All of it comes out of one pass
// over the row:
//   m = max_v z_v, a = lowest index attaining m, S = sum_v 2^((z_v - m) * log2(e)/T),
//   and p(child token) = 2^((z_t - m) * log2(e)/T) / S for every child of the row's node.
// The running max is updated per 16-byte vector (8 bf16): a vector whose NaN-propagating max
// does not exceed the running max costs 4 packed max instructions; otherwise (rare: O(log n)
// times per thread) the sum is rescaled. Elements are visited in increasing index order per
// thread, so a strict '>' keeps the lowest index; partial results merge lowest-index-first.
// The stream is HBM-bound: 16-byte read-only loads, 4 in flight per thread, 256 threads per
// CTA and 6 CTAs per SM (16 KiB of loads in flight per CTA).
// The CTA splits the row into kRowChunks contiguous chunks, each streamed by its own group of
// warps (threads interleaved, so one load instruction of a group covers contiguous memory).
// For 16-byte aligned rows the chunks start on 256-element sub-tile boundaries, and in
// sampling mode each chunk's (max, sum) is stored: the walk then locates the chunk holding
// its inverse-CDF draw from these partials and re-reads only that chunk.

#include <cfloat>

#include "row_pass.cuh"
#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

using namespace rowpass;


constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// The statistics of one row: row blockIdx.x (blockIdx.x - first for the second set of a
// paired launch), or, with SPLIT > 1, piece blockIdx.x % SPLIT of row blockIdx.x / SPLIT.
template <int DT, int MODE, bool SECOND, int SPLIT = 1, int kUnroll = SPEC_ROW_UNROLL>
__device__ __forceinline__ void row_stats_row(const RowStatsParams P, int first) {
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kEpv = 16 / kEsz;   // elements per 16-byte vector
    constexpr int kChunksPerCta = kRowChunks / SPLIT;
    constexpr int kGroup = kThreads / kChunksPerCta;         // threads per chunk
    constexpr int kWarpsPerGroup = kWarps / kChunksPerCta;
    static_assert(kChunksPerCta * SPLIT == kRowChunks && kWarpsPerGroup >= 1, "row split");
    const int cta = SECOND ? (int)blockIdx.x - first : (int)blockIdx.x;
    const int row = cta / SPLIT, piece = cta - row * SPLIT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // debug builds: the request a violation is charged to (clamped into the batch)
    int32_t *const dbg = P.dbg;
    const int dbg_b = min(row, P.rows - 1) / P.N;
    if (!dbg_check(row < P.rows, dbg, dbg_b, DBG_INDEX)) return;
    const int64_t V = P.V;
    const char *rowp = reinterpret_cast<const char *>(P.x) + (size_t)row * (size_t)V * kEsz;

    __shared__ Part sh_part[kWarps];
    __shared__ int sh_leaf;

    // Children of this row's node (warp 0): lane handles nodes lane and lane + 32.
    const bool gather = P.pc != nullptr;
    const int N = P.N;
    const int b = row / N, n = row - b * N;
    const int nb = node_budget(P.n_active, b, N);   // nodes >= nb do not exist in this call
    if (n >= nb) return;
    int child[2] = {-1, -1};
    float zc[2] = {0.f, 0.f};
    if (warp == 0 && (gather || P.skip_leaves)) {
        bool any = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = lane + 32 * h;
            if (c >= 1 && c < nb && P.parent[(size_t)b * N + c] == n) {
                any = true;
                const int t = P.tok[(size_t)b * N + c];
                if (t >= 0 && t < V && dbg_check(c < N, dbg, dbg_b, DBG_INDEX)) {
                    child[h] = c;
                    if (gather) zc[h] = load_elem<DT>(rowp, t);   // prefetch, used at the end
                }
            }
        }
        if (P.skip_leaves) {
            const unsigned bal = __ballot_sync(0xffffffffu, any);
            if (lane == 0) sh_leaf = bal == 0;
        }
    }
    if (P.skip_leaves) {
        __syncthreads();
        if (sh_leaf) return;
    }

    const float k = P.k;
    Acc a = acc_init();

    // Split the row into a scalar head up to 16-byte alignment, vectors, and a scalar tail;
    // thread group g takes vectors [row_chunk_vec(g), row_chunk_vec(g + 1)), group 0 the head
    // and the last group the tail.
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
    int64_t head = (int64_t)((16 - (addr & 15)) & 15) / kEsz;
    if (head > V) head = V;
    const int nv = (int)((V - head) / kEpv);
    const int64_t tail0 = head + (int64_t)nv * kEpv;
    const bool aligned = head == 0;
    const int g = piece * kChunksPerCta + tid / kGroup, gt = tid % kGroup;   // chunk, rank
    const int v1 = row_chunk_vec(g + 1, nv, V, aligned, kEpv);
    if (g == 0 && gt < head && dbg_check(gt < V, dbg, dbg_b, DBG_INDEX))
        proc_scalar<MODE>(a, load_elem<DT>(rowp, gt), gt, k);

    const uint4 *vb = reinterpret_cast<const uint4 *>(rowp + head * kEsz);
    int i = row_chunk_vec(g, nv, V, aligned, kEpv) + gt;
    for (; i + (kUnroll - 1) * kGroup < v1; i += kUnroll * kGroup) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            w[u] = ldg_checked(vb, i + u * kGroup, nv, dbg, dbg_b);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int e0 = (int)head + (i + u * kGroup) * kEpv;
            if (DT == 1)
                proc_bf16<MODE>(a, w[u], e0, k);
            else
                proc_f32<MODE>(a, w[u], e0, k);
        }
    }
    for (; i < v1; i += kGroup) {
        const uint4 w = ldg_checked(vb, i, nv, dbg, dbg_b);
        const int e0 = (int)head + i * kEpv;
        if (DT == 1)
            proc_bf16<MODE>(a, w, e0, k);
        else
            proc_f32<MODE>(a, w, e0, k);
    }
    if (g == kRowChunks - 1 && tail0 + gt < V) {
        const int idx = (int)(tail0 + gt);
        proc_scalar<MODE>(a, load_elem<DT>(rowp, idx), idx, k);
    }

    // CTA reduction: warps, then warp 0 over the warp results (fixed order: deterministic).
    Part p{a.m, a.s0 + a.s1, a.arg, a.flags};
    p = warp_merge<MODE>(p, k);
    if (lane == 0) sh_part[warp] = p;
    __syncthreads();
    if (warp != 0) return;
    p = lane < kWarps ? sh_part[lane] : Part{-INFINITY, 0.f, kNone, 0};
    // warps of one chunk first (consecutive lanes), then across chunks
#pragma unroll
    for (int o = 1; o < kWarpsPerGroup; o <<= 1) p = merge<MODE>(p, shfl_part(p, o), k);
    if (MODE == ROW_SAMPLE && P.chunk && aligned && lane < kWarps && lane % kWarpsPerGroup == 0 &&
        dbg_check(piece * kChunksPerCta + lane / kWarpsPerGroup < kRowChunks, dbg, dbg_b,
                  DBG_INDEX))
        P.chunk[(size_t)row * kRowChunks + piece * kChunksPerCta + lane / kWarpsPerGroup] =
            make_float2(p.m, p.s);
#pragma unroll
    for (int o = kWarpsPerGroup; o < 32; o <<= 1) p = merge<MODE>(p, shfl_part(p, o), k);
    if (SPLIT > 1) {
        // Publish this piece's statistics; the row's last CTA to arrive merges all of them (a
        // fixed merge tree over the pieces, so the result does not depend on which CTA is
        // last) and resets the row's counter for the next launch.
        RowPart *parts = P.piece + (size_t)row * SPLIT;
        int last = 0;
        if (lane == 0) {
            parts[piece] = RowPart{p.m, p.s, p.arg, p.flags};
            __threadfence();
            const int old = atomicAdd(&P.count[row], 1);
            // the counter is zero between launches, so the arrivals see 0 .. SPLIT-1
            dbg_check(old >= 0 && old < SPLIT, dbg, dbg_b, DBG_ARRIVAL);
            last = old == SPLIT - 1;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence();
        p = Part{-INFINITY, 0.f, kNone, 0};
        if (lane < SPLIT) {
            const volatile RowPart *vp = parts + lane;   // written by other CTAs: bypass L1
            p = Part{vp->m, vp->s, vp->arg, vp->flags};
        }
        // full butterfly: every lane of warp 0 needs the row's statistics (child gathers)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) p = merge<MODE>(p, shfl_part(p, o), k);
        if (lane == 0) P.count[row] = 0;
    }

    if (MODE != ROW_PROBS) {
        if (p.m == INFINITY) p.flags |= F_POSINF;
        if (p.m == -INFINITY) p.flags |= F_ALLNEG;
    }
    if (lane == 0) {
        if (P.m) P.m[row] = p.m;
        if (P.s) P.s[row] = p.s;
        if (P.arg) P.arg[row] = p.arg == kNone ? 0 : p.arg;
        P.flags[row] = p.flags;
    }
    if (gather) {
        const float negm = p.m == -INFINITY ? 0.f : -p.m;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (child[h] < 0) continue;
            float v;
            if (MODE == ROW_PROBS)
                v = zc[h];
            else
                v = P.pc_normalized ? ex2((zc[h] + negm) * k) / p.s : ex2((zc[h] + negm) * k);
            P.pc[(size_t)b * N + child[h]] = v;
        }
    }
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kThreads, kRowCtasPerSm) row_stats_kernel(RowStatsParams P) {
    grid_dep_wait();     // the logits (and the tree) come from earlier kernels
    grid_dep_launch();   // the walk may start launching: it waits for this grid's results
    row_stats_row<DT, MODE, false>(P, 0);
}

// Target rows and dense-draft rows in one launch (the first A.rows CTAs take the target rows):
// both sets are streamed at once instead of one launch after the other.
template <int DT1, int MODE1, int DT2, int MODE2>
__global__ void __launch_bounds__(kThreads, SPEC_PAIR_MIN_CTAS)
    row_stats_pair_kernel(RowStatsParams A, RowStatsParams B) {
    grid_dep_wait();
    grid_dep_launch();
    if ((int)blockIdx.x < A.rows)
        row_stats_row<DT1, MODE1, false, 1, SPEC_PAIR_UNROLL>(A, 0);
    else
        row_stats_row<DT2, MODE2, true, 1, SPEC_PAIR_UNROLL>(B, A.rows);
}

template <int DT1, int DT2, int MODE2>
cudaError_t launch_pair(const RowStatsParams &a, const RowStatsParams &b, cudaStream_t st) {
    return launch_dependent(row_stats_pair_kernel<DT1, ROW_SAMPLE, DT2, MODE2>,
                            dim3(a.rows + b.rows), dim3(kThreads), 0, st, a, b);
}

template <int DT1>
cudaError_t launch_pair_d(const RowStatsParams &a, const RowStatsParams &b, int dtype2,
                          int mode2, cudaStream_t st) {
    if (mode2 == ROW_PROBS) return launch_pair<DT1, 0, ROW_PROBS>(a, b, st);
    if (dtype2 == 1) return launch_pair<DT1, 1, ROW_SAMPLE>(a, b, st);
    return launch_pair<DT1, 0, ROW_SAMPLE>(a, b, st);
}

// Small batches: SPLIT CTAs per row (each streaming kRowChunks / SPLIT chunks) so that one
// wave of CTAs covers the GPU.
template <int DT, int MODE, int SPLIT>
__global__ void __launch_bounds__(kThreads, kSplitCtasPerSm)
    row_stats_split_kernel(RowStatsParams P) {
    grid_dep_wait();
    grid_dep_launch();
    row_stats_row<DT, MODE, false, SPLIT, SPEC_SPLIT_UNROLL>(P, 0);
}

template <int DT, int MODE>
cudaError_t launch(const RowStatsParams &p, cudaStream_t st) {
    if (p.piece && p.count) {
        const dim3 block(kThreads);
        if (p.split == 8)
            return launch_dependent(row_stats_split_kernel<DT, MODE, 8>, dim3(p.rows * 8), block,
                                    0, st, p);
        if (p.split == 4)
            return launch_dependent(row_stats_split_kernel<DT, MODE, 4>, dim3(p.rows * 4), block,
                                    0, st, p);
        if (p.split == 2)
            return launch_dependent(row_stats_split_kernel<DT, MODE, 2>, dim3(p.rows * 2), block,
                                    0, st, p);
    }
    return launch_dependent(row_stats_kernel<DT, MODE>, dim3(p.rows), dim3(kThreads), 0, st, p);
}

}  // namespace

cudaError_t launch_row_stats_pair(const RowStatsParams &target, int dtype, const RowStatsParams &draft,
                                  int draft_dtype, int draft_mode, cudaStream_t st) {
    if (target.rows + draft.rows <= 0) return cudaSuccess;
    if (dtype == 1) return launch_pair_d<1>(target, draft, draft_dtype, draft_mode, st);
    return launch_pair_d<0>(target, draft, draft_dtype, draft_mode, st);
}

cudaError_t launch_row_stats(const RowStatsParams &p, int dtype, int mode, cudaStream_t st) {
    if (p.rows <= 0) return cudaSuccess;
    if (dtype == 1) {
        if (mode == ROW_GREEDY) return launch<1, ROW_GREEDY>(p, st);
        if (mode == ROW_SAMPLE) return launch<1, ROW_SAMPLE>(p, st);
        return cudaErrorInvalidValue;
    }
    if (mode == ROW_GREEDY) return launch<0, ROW_GREEDY>(p, st);
    if (mode == ROW_SAMPLE) return launch<0, ROW_SAMPLE>(p, st);
    return launch<0, ROW_PROBS>(p, st);
}

}  // namespace specv
