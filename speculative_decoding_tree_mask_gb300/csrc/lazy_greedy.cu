// Greedy verification that reads only the rows on the accepted path.
//
// EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput",
// commit 4b728e2: greedy decoding keeps the argmax path. The walk needs the argmax of the
// current node's row only, so one CTA per request streams the root's row, moves to the first
// child whose token equals the argmax, streams that child's row, and so on: at most
// depth + 1 rows per request instead of all N. The per-element arithmetic is the same as
// the row-statistics kernel's; results equal spec_verify_greedy's bit for bit.

#include "row_pass.cuh"
#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

struct LazySmem {
    int par[kMaxN], tok[kMaxN], path[kMaxN];
    int st, next;
    int dbgv;   // debug builds: violation bits found by this CTA
    rowpass::Part part[kWarps], part_out;
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) lazy_greedy_kernel(LazyGreedyParams P) {
    constexpr int kEsz = DT == 1 ? 2 : 4;
    __shared__ LazySmem sm;
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int N = P.N;
    const size_t base = (size_t)b * N;
    const int nb = node_budget(P.n_active, b, N);   // nodes >= nb do not exist in this call
    if (tid < N) {
        sm.par[tid] = tid < nb ? P.parent[base + tid] : -2;
        sm.tok[tid] = tid < nb ? P.tok[base + tid] : -1;
    }
    __syncthreads();
    if (warp == 0) {
        bool bp = false, bt = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            if (i < nb) {
                const int p = sm.par[i];
                bp |= i == 0 ? p != -1 : (p < 0 || p >= i);
                if (i >= 1) bt |= sm.tok[i] < 0 || sm.tok[i] >= P.V;
            }
        }
        const int st = nb == 0 ? SPEC_REQ_BAD_BUDGET
                       : __any_sync(full, bp) ? SPEC_REQ_BAD_PARENT
                       : __any_sync(full, bt) ? SPEC_REQ_BAD_TOKEN
                                              : SPEC_REQ_OK;
        if (lane == 0) sm.st = st;
    }
    if (tid == 0) sm.dbgv = 0;
    __syncthreads();

    int st = sm.st, node = 0, L = 0, a = -1;
    while (st == SPEC_REQ_OK) {
        const char *row = reinterpret_cast<const char *>(P.logits) + (base + node) * (size_t)P.V * kEsz;
        const rowpass::Part p = rowpass::cta_row_stats<DT, ROW_GREEDY, kThreads, 4>(
            row, P.V, 0.f, sm.part, &sm.part_out, &sm.dbgv);
        if (p.flags) {
            st = SPEC_REQ_BAD_ROW;
            break;
        }
        a = p.arg;
        if (warp == 0) {
            const unsigned m0 = __ballot_sync(
                full, lane >= 1 && lane < N && sm.par[lane] == node && sm.tok[lane] == a);
            const unsigned m1 = __ballot_sync(
                full, lane + 32 < N && sm.par[lane + 32] == node && sm.tok[lane + 32] == a);
            if (lane == 0) sm.next = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : -1);
        }
        __syncthreads();
        const int next = sm.next;
        if (next < 0) break;
        if (kDebug && !(L < N - 1 && next >= 1 && next < N)) {
            if (tid == 0) sm.dbgv |= DBG_WALK;
            break;
        }
        if (tid == 0) sm.path[L] = next;
        ++L;
        node = next;
        __syncthreads();
    }
    __syncthreads();
    if constexpr (kDebug) {
        // the accepted path is a chain of parent links and the bonus a token
        if (tid == 0) {
            int v = sm.dbgv;
            if (st == SPEC_REQ_OK) {
                int prev = 0;
                for (int j = 0; j < L; ++j) {
                    const int nd = sm.path[j];
                    if (nd < 1 || nd >= N || sm.par[nd] != prev) v |= DBG_WALK;
                    prev = nd >= 0 && nd < N ? nd : 0;
                }
                if (!(a >= 0 && a < P.V)) v |= DBG_WALK;
            }
            if (v && P.dbg) atomicOr(P.dbg + b, v);
            sm.dbgv = v;
        }
        __syncthreads();
        if (sm.dbgv) st = SPEC_REQ_INTERNAL;
    }
    for (int j = tid; j < N; j += kThreads) {
        int ot = -1, kv = -1;
        if (st == SPEC_REQ_OK) {
            if (j < L)
                ot = sm.tok[sm.path[j]];
            else if (j == L)
                ot = a;
            if (j == 0)
                kv = 0;
            else if (j <= L)
                kv = sm.path[j - 1];
        }
        P.out.out_tokens[base + j] = ot;
        P.out.kv_commit[base + j] = kv;
    }
    if (tid == 0) {
        P.out.accept_len[b] = st ? 0 : L;
        P.out.bonus[b] = st ? -1 : a;
        P.out.status[b] = st;
    }
}

}  // namespace

cudaError_t launch_lazy_greedy(const LazyGreedyParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    if (p.dtype == 1)
        lazy_greedy_kernel<1><<<p.B, kThreads, 0, st>>>(p);
    else
        lazy_greedy_kernel<0><<<p.B, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
