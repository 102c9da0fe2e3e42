// Adaptive node budget: one controller update per verify step, on the device.
//
// IluvatarLabs/vllm PR #3 "SCV vectorized masking", adaptive mode: the number of speculative
// tokens verified per step is adjusted from recent acceptance ratios so that the ratio stays
// near a target, and the mask work runs from captured CUDA graphs. Here the ratio of a step
// is (accepted nodes) / (the most that could have been accepted: the deepest node within each
// request's budget), summed over the usable requests; a moving average of it moves the budget
// up or down by a fixed step outside a dead band. Reading the budget back from device memory
// lets a graph captured once follow every update.
//
// One CTA: a thread per request computes that request's deepest node among nodes 0..n-1 from
// the parent array (parent[i] < i, so one forward sweep suffices), the integer sums are
// reduced exactly, and thread 0 evaluates the float64 update with explicitly rounded
// operations in a fixed order (no contraction), so the state is reproducible bit for bit.

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) budget_update_kernel(BudgetParams P) {
    __shared__ long long sh_a[kWarps], sh_d[kWarps];
    __shared__ int sh_budget;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = P.N;

    long long acc = 0, deep = 0;
    for (int b = tid; b < P.B; b += kThreads) {
        if (P.status[b] != SPEC_REQ_OK) continue;
        const int n = P.n_active[b];
        if (n < 1 || n > N) continue;
        const int32_t *par = P.parent + (size_t)b * N;
        unsigned char depth[kMaxN];
        depth[0] = 0;
        int dmax = 0;
        bool ok = par[0] == -1;
        for (int i = 1; i < n && ok; ++i) {
            const int p = par[i];
            if (p < 0 || p >= i) {
                ok = false;
                break;
            }
            depth[i] = (unsigned char)(depth[p] + 1);
            dmax = max(dmax, (int)depth[i]);
        }
        if (!ok) continue;
        acc += P.accept_len[b];
        deep += dmax;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc += __shfl_down_sync(0xffffffffu, acc, o);
        deep += __shfl_down_sync(0xffffffffu, deep, o);
    }
    if (lane == 0) {
        sh_a[warp] = acc;
        sh_d[warp] = deep;
    }
    __syncthreads();   // every read of n_active is done before it is rewritten below
    if (tid == 0) {
        long long A = 0, D = 0;
        for (int w = 0; w < kWarps; ++w) {
            A += sh_a[w];
            D += sh_d[w];
        }
        const spec_budget_params &q = P.prm;
        spec_budget_state s = *P.state;
        int k = min(max(s.budget, q.n_min), q.n_max);
        if (D > 0) {
            const double ratio = __ddiv_rn((double)A, (double)D);
            const double ema = __dadd_rn(__dmul_rn(__dsub_rn(1.0, q.alpha), s.ema),
                                         __dmul_rn(q.alpha, ratio));
            s.ema = ema;
            s.steps += 1;
            if (ema > __dadd_rn(q.target, q.band))
                k = min(k + q.step, q.n_max);
            else if (ema < __dsub_rn(q.target, q.band))
                k = max(k - q.step, q.n_min);
        }
        s.budget = k;
        *P.state = s;
        sh_budget = k;
    }
    __syncthreads();
    const int k = sh_budget;
    for (int b = tid; b < P.B; b += kThreads) P.n_active[b] = k;
}

}  // namespace

cudaError_t launch_budget_update(const BudgetParams &p, cudaStream_t st) {
    budget_update_kernel<<<1, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
