// Tree-attention mask: per-node ancestor bitmask and depth, one warp per request.
//
// EmbodiInfer PR #11 (commit 4b728e2) verifies all trie nodes in one tree-attention forward:
// node i may attend to the committed context, to itself and to its ancestors. With the parent
// array in topological order the ancestor set is closed under "ancestor of my parent", so it
// is built by pointer jumping: anc[i] = {i}, hop[i] = parent[i]; each round
// anc[i] |= anc[hop[i]], hop[i] = hop[hop[i]] doubles the covered distance, and 6 rounds cover
// depth <= 63. Depth is the number of ancestors: popcount(anc[i]) - 1.

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kWarpsPerCta = 4;

__global__ void __launch_bounds__(32 * kWarpsPerCta)
    tree_mask_kernel(const int32_t *__restrict__ parent, int B, int N,
                     uint64_t *__restrict__ anc_out, int32_t *__restrict__ depth_out,
                     int32_t *__restrict__ status) {
    __shared__ unsigned long long s_anc[kWarpsPerCta][kMaxN];
    __shared__ int s_hop[kWarpsPerCta][kMaxN];
    grid_dep_launch();   // a verify call after this one may start launching (it waits for us)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerCta + warp;
    if (b >= B) return;
    const int32_t *par = parent + (size_t)b * N;

    bool bad = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < N) {
            const int p = par[i];
            bad |= i == 0 ? p != -1 : (p < 0 || p >= i);
            s_anc[warp][i] = 1ull << i;
            s_hop[warp][i] = p;
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    bool viol = false;   // debug builds: a hop outside the request's nodes
    if (!bad) {
        __syncwarp();
#pragma unroll 1
        for (int round = 0; round < 6; ++round) {
            unsigned long long na[2];
            int nh[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                na[h] = 0;
                nh[h] = -1;
                if (i < N) {
                    const int j = s_hop[warp][i];
                    na[h] = s_anc[warp][i];
                    if (kDebug && j >= N) {
                        viol = true;
                    } else if (j >= 0) {
                        na[h] |= s_anc[warp][j];
                        nh[h] = s_hop[warp][j];
                    }
                }
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                if (i < N) {
                    s_anc[warp][i] = na[h];
                    s_hop[warp][i] = nh[h];
                }
            }
            __syncwarp();
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < N) {
            const unsigned long long a = bad ? 0ull : s_anc[warp][i];
            anc_out[(size_t)b * N + i] = a;
            depth_out[(size_t)b * N + i] = bad ? -1 : __popcll(a) - 1;
        }
    }
    if (kDebug) viol = __any_sync(0xffffffffu, viol);
    if (lane == 0) status[b] = bad ? 1 : (viol ? SPEC_REQ_INTERNAL : 0);
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                             int32_t *status, cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    const int grid = (B + kWarpsPerCta - 1) / kWarpsPerCta;
    tree_mask_kernel<<<grid, 32 * kWarpsPerCta, 0, st>>>(parent, B, N, anc, depth, status);
    return cudaGetLastError();
}

}  // namespace specv
