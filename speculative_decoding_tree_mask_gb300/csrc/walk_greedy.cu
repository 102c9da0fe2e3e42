// Greedy tree walk and accepted-path compaction.
//
// EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput",
// commit 4b728e2: greedy decoding keeps the argmax path. From the root, the walk moves to the
// first child (ascending node index) whose draft token equals the argmax of the current
// node's row and stops when none does; the bonus token is the argmax at the stop node.
//
// One warp per request: the request's parents, tokens and per-row argmax / flags (N <= 64)
// sit in two registers per lane, and the children of the current node are found with one
// ballot per half of the tree.

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kGreedyWarps = 4;

__global__ void __launch_bounds__(32 * kGreedyWarps) walk_greedy_kernel(GreedyWalkParams P) {
    const unsigned full = 0xffffffffu;
    grid_dep_wait();   // row statistics of the kernel before
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kGreedyWarps + warp;
    if (b >= P.B) return;
    const int N = P.N;
    const size_t base = (size_t)b * N;
    const int nb = node_budget(P.n_active, b, N);   // nodes >= nb do not exist in this call

    int par[2], tk[2], ag[2], fl[2];
    bool bad_par = false, bad_tok = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < nb) {
            par[h] = P.parent[base + i];
            tk[h] = P.tok[base + i];
            ag[h] = P.arg[base + i];
            fl[h] = P.flags[base + i];
            bad_par |= i == 0 ? par[h] != -1 : (par[h] < 0 || par[h] >= i);
            bad_tok |= i >= 1 && (tk[h] < 0 || tk[h] >= P.V);
        } else {
            par[h] = -2;
            tk[h] = -1;
            ag[h] = 0;
            fl[h] = 0;
        }
    }
    int st = nb == 0                        ? SPEC_REQ_BAD_BUDGET
             : __any_sync(full, bad_par) ? SPEC_REQ_BAD_PARENT
             : __any_sync(full, bad_tok) ? SPEC_REQ_BAD_TOKEN
                                         : SPEC_REQ_OK;
    bool viol = false;   // debug builds: a check of this walk failed

    int L = 0, node = 0, a = -1;
    int pth0 = -1, pth1 = -1;   // path[j] lives in lane j % 32, slot j / 32
    if (st == 0) {
        for (;;) {
            const int src = node & 31;
            const int f = __shfl_sync(full, node < 32 ? fl[0] : fl[1], src);
            if (f != 0) {
                st = 3;
                break;
            }
            a = __shfl_sync(full, node < 32 ? ag[0] : ag[1], src);
            const unsigned m0 = __ballot_sync(full, lane >= 1 && par[0] == node && tk[0] == a);
            const unsigned m1 = __ballot_sync(full, par[1] == node && tk[1] == a);
            int c;
            if (m0)
                c = __ffs(m0) - 1;
            else if (m1)
                c = 32 + __ffs(m1) - 1;
            else
                break;
            if (!dbg_check(c >= 1 && c < nb && L < N - 1, P.dbg, b, DBG_WALK)) {
                viol = true;
                break;
            }
            if (lane == (L & 31)) {
                if (L < 32)
                    pth0 = c;
                else
                    pth1 = c;
            }
            ++L;
            node = c;
        }
    }

    // Compaction: out_tokens = tokens of path[0..L) then the bonus; kv_commit = 0, path.
    const int prev0 = __shfl_sync(full, pth0, (lane + 31) & 31);
    const int prev1 = __shfl_sync(full, pth1, (lane + 31) & 31);
    if constexpr (kDebug) {
        // The accepted path is a chain of parent links from the root, the bonus a token, and
        // no row statistics of this request failed a check.
        if (st == 0) {
            bool bad = !(a >= 0 && a < P.V);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = lane + 32 * h;
                const int nd = h == 0 ? pth0 : pth1;
                const int pv = j == 0 ? 0 : (h == 0 ? prev0 : (lane == 0 ? prev0 : prev1));
                const int pa = __shfl_sync(full, par[0], nd & 31);
                const int pb = __shfl_sync(full, par[1], nd & 31);
                if (j < L) bad |= nd < 1 || nd >= nb || (nd < 32 ? pa : pb) != pv;
            }
            if (__any_sync(full, bad)) {
                dbg_check(false, P.dbg, b, DBG_WALK);
                viol = true;
            }
        }
        if (P.dbg && P.dbg[b] != 0) viol = true;
        if (viol) st = SPEC_REQ_INTERNAL;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int j = lane + 32 * h;
        const int pj = h == 0 ? pth0 : pth1;
        const int ta = __shfl_sync(full, tk[0], pj & 31);
        const int tb = __shfl_sync(full, tk[1], pj & 31);
        const int prev = h == 0 ? prev0 : (lane == 0 ? prev0 : prev1);
        if (j < N) {
            int ot = -1, kv = -1;
            if (st == 0) {
                if (j < L)
                    ot = pj < 32 ? ta : tb;
                else if (j == L)
                    ot = a;
                if (j == 0)
                    kv = 0;
                else if (j <= L)
                    kv = prev;
            }
            P.out.out_tokens[base + j] = ot;
            P.out.kv_commit[base + j] = kv;
        }
    }
    if (lane == 0) {
        P.out.accept_len[b] = st ? 0 : L;
        P.out.bonus[b] = st ? -1 : a;
        P.out.status[b] = st;
    }
}

}  // namespace

cudaError_t launch_walk_greedy(const GreedyWalkParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    const int grid = (p.B + kGreedyWarps - 1) / kGreedyWarps;
    return launch_dependent(walk_greedy_kernel, dim3(grid), dim3(32 * kGreedyWarps), 0, st, p);
}

}  // namespace specv
