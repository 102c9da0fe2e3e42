// Greedy verification that allocates nothing (spec_verify_greedy_noalloc).
//
// spec_verify_greedy keeps its per-row scratch (the argmax and flags of every (request, node)
// row, written by the row-statistics kernel and read by the walk) in the workspace that
// spec_verify_init obtains with cudaMalloc. This variant keeps that scratch in a file-scope
// static device array instead, so a caller that cannot allocate device memory can still
// verify. The kernels are the same ones the handle path launches.

#include <mutex>

#include <cuda.h>

#include "spec_internal.h"
#include "spec_verify.h"

using namespace specv;

// argmax of SPEC_NOALLOC_MAX_ROWS rows, then their flags: 2 * 16384 * 4 bytes = 128 KiB
// (the debug build adds one violation word per request, 64 KiB more). Every GPU that loads
// this library holds the array until the process exits.
#ifdef SPEC_DEBUG
constexpr int kScratchWords = 3 * SPEC_NOALLOC_MAX_ROWS;
#else
constexpr int kScratchWords = 2 * SPEC_NOALLOC_MAX_ROWS;
#endif
static __device__ __align__(256) int32_t g_noalloc_scratch[kScratchWords];

namespace {

constexpr int kMaxDevices = 64;

// The array's address belongs to the context the module was loaded in: after
// cudaDeviceReset, or under another driver-API context made current on the same device, the
// module is loaded again at another address. So the cached address is kept per device
// together with the ID of the context it was looked up in, and looked up again whenever the
// current context's ID differs.
struct ScratchEntry {
    unsigned long long ctx = 0;
    int32_t *addr = nullptr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices];

// Driver calls that read the current context's ID, resolved through the runtime (so the
// library needs no link-time dependency on the driver library).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

bool resolve_driver_calls() {
    if (g_ctx_get_current && g_ctx_get_id) return true;
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) !=
            cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b) {
        cudaGetLastError();
        return false;
    }
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
    return true;
}

// ID of the current context; false when no context is current yet.
bool current_context_id(unsigned long long *id) {
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context of device `dev`. In host code
// the array's name is only a host-side stand-in, so the address is looked up with that
// context current (cudaGetSymbolAddress) and cached with the context's ID.
int scratch_address(int dev, int32_t **out) {
    if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!resolve_driver_calls()) return SPEC_ERR_CUDA;
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    ScratchEntry &e = g_scratch[dev];
    if (have_id && e.addr != nullptr && e.ctx == id) {
        *out = e.addr;
        return SPEC_OK;
    }
    // Looking the symbol up also makes the runtime's context current if none was yet.
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    if (!have_id && !current_context_id(&id)) return SPEC_ERR_CUDA;
    e.ctx = id;
    e.addr = static_cast<int32_t *>(p);
    *out = e.addr;
    return SPEC_OK;
}

// The logits must be memory of the current device (they are streamed by the row-statistics
// kernel, launched there): device memory of another GPU is refused rather than read
// through an address that is not valid on this one.
bool on_device(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
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

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
    if (!on_device(logits, dev)) return SPEC_ERR_ARG;
    int32_t *scratch = nullptr;
    const int rc = scratch_address(dev, &scratch);
    if (rc != SPEC_OK) return rc;
    int32_t *arg = scratch;
    int32_t *flags = scratch + SPEC_NOALLOC_MAX_ROWS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Every row's argmax and flags are written by the first kernel before the walk reads
    // them, so nothing left in the array by an earlier call needs clearing.
    int32_t *dbg = nullptr;
#ifdef SPEC_DEBUG
    // debug builds: the requests' violation words, zeroed for this call
    dbg = scratch + 2 * SPEC_NOALLOC_MAX_ROWS;
    if (cudaMemsetAsync(dbg, 0, sizeof(int32_t) * (size_t)B, st) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_CUDA;
    }
#endif
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
    rp.dbg = dbg;
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
    gp.dbg = dbg;
    if (launch_walk_greedy(gp, st) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}
