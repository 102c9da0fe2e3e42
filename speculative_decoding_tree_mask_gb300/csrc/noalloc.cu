// Greedy verification that allocates nothing (spec_verify_greedy_noalloc).
//
// spec_verify_greedy keeps its per-row scratch (the argmax and flags of every (request, node)
// row, written by the row-statistics kernel and read by the walk) in the workspace that
// spec_verify_init obtains with cudaMalloc. This variant keeps that scratch in a file-scope
// static device array instead, so a caller that cannot allocate device memory can still
// verify. The kernels are the same ones the handle path launches.

#include <mutex>

#include "spec_internal.h"
#include "spec_verify.h"

using namespace specv;

// argmax of SPEC_NOALLOC_MAX_ROWS rows, then their flags: 2 * 16384 * 4 bytes = 128 KiB.
// Every GPU that loads this library holds the array until the process exits.
static __device__ __align__(256) int32_t g_noalloc_scratch[2 * SPEC_NOALLOC_MAX_ROWS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the array's name
// is only a host-side stand-in, so the address is looked up once per device (with that
// device current) and cached.
int scratch_address(int32_t **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SPEC_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return SPEC_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int spec_verify_greedy_noalloc(const void *logits, int dtype, int B, int N, int64_t V,
                                          const int32_t *draft_token, const int32_t *parent,
                                          int32_t *accept_len, int32_t *out_tokens,
                                          int32_t *kv_commit, int32_t *bonus, int32_t *status,
                                          void *stream) {
    if (B < 0 || N < 1 || N > kMaxN || V < 1 || V > (int64_t(1) << 21)) return SPEC_ERR_ARG;
    if ((int64_t)B * N > SPEC_NOALLOC_MAX_ROWS) return SPEC_ERR_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    if (!logits || !draft_token || !parent || !accept_len || !out_tokens || !kv_commit ||
        !bonus || !status)
        return SPEC_ERR_ARG;
    if (!aligned_to(logits, dtype == SPEC_BF16 ? 2 : 4)) return SPEC_ERR_ARG;
    const void *ints[] = {draft_token, parent, accept_len, out_tokens, kv_commit, bonus, status};
    for (const void *p : ints)
        if (!aligned_to(p, 4)) return SPEC_ERR_ARG;

    int32_t *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SPEC_OK) return rc;
    int32_t *arg = scratch;
    int32_t *flags = scratch + SPEC_NOALLOC_MAX_ROWS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Every row's argmax and flags are written by the first kernel before the walk reads
    // them, so nothing left in the array by an earlier call needs clearing.
    RowStatsParams rp{};
    rp.x = logits;
    rp.V = V;
    rp.rows = B * N;
    rp.N = N;
    rp.k = 0.f;
    rp.m = nullptr;
    rp.s = nullptr;
    rp.arg = arg;
    rp.flags = flags;
    if (launch_row_stats(rp, dtype, ROW_GREEDY, st) != cudaSuccess) return SPEC_ERR_CUDA;

    GreedyWalkParams gp;
    gp.B = B;
    gp.N = N;
    gp.V = V;
    gp.parent = parent;
    gp.tok = draft_token;
    gp.arg = arg;
    gp.flags = flags;
    gp.out.accept_len = accept_len;
    gp.out.out_tokens = out_tokens;
    gp.out.kv_commit = kv_commit;
    gp.out.bonus = bonus;
    gp.out.status = status;
    if (launch_walk_greedy(gp, st) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}
