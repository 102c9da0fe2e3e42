// C ABI of the verification library (declared in include/spec_verify.h): handle and
// workspace, host-side argument checks, kernel orchestration and per-kernel timing.

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <new>

#include "spec_internal.h"
#include "spec_verify.h"

// Built with SPEC_NVTX, every entry point of the ABI is an NVTX range named after it, so a
// timeline profiler shows the host side of each call around its kernels. Otherwise the
// ranges compile to nothing.
#ifdef SPEC_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
}  // namespace
#define SPEC_RANGE(name) NvtxRange spec_range_(name)
#else
#define SPEC_RANGE(name) ((void)0)
#endif

using namespace specv;

namespace {

constexpr int kMaxRecords = 16384;
constexpr int64_t kMaxV = int64_t(1) << 21;
constexpr float kLog2eF = 1.4426950408889634f;

}  // namespace

struct spec_ctx {
    int device = 0;
    int max_B = 0, max_N = 0;
    int64_t max_V = 0;
    void *ws = nullptr;
    float *m = nullptr, *s = nullptr, *pc = nullptr, *mq = nullptr, *sq = nullptr,
          *qc = nullptr;
    int32_t *arg = nullptr, *flags = nullptr, *dflags = nullptr;
    float2 *chunk = nullptr;              // row-chunk partials of the target rows
    RowPart *piece = nullptr;             // small batches: per-piece row statistics
    int32_t *count = nullptr;             // ... and per-row arrivals (zero between calls)
    int32_t *dbg = nullptr;               // debug builds: violation bits per request [max_B]
    int inject_row = -1, inject_value = 0;   // debug builds: one armed counter injection
    int slots = 0;                        // CTAs of the split row-statistics kernel in a wave
    int sms = 0;                          // streaming multiprocessors of the device
    const int32_t *n_active = nullptr;   // node budget set by spec_set_node_budget
    bool prof = false;
    bool ev_ready = false;
    int nrec = 0;
    cudaEvent_t ev[2 * kMaxRecords];
    int cls[kMaxRecords];
};

namespace {

// Makes the handle's device current for the duration of a call and restores the caller's.
class DeviceScope {
  public:
    explicit DeviceScope(int dev) {
        ok_ = cudaGetDevice(&prev_) == cudaSuccess;
        if (ok_ && prev_ != dev) ok_ = cudaSetDevice(dev) == cudaSuccess;
        switched_ = ok_ && prev_ != dev;
    }
    ~DeviceScope() {
        if (switched_) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

  private:
    int prev_ = 0;
    bool ok_ = false, switched_ = false;
};

template <typename F>
int timed(spec_handle h, int cls, cudaStream_t st, F &&launch) {
    int slot = -1;
    if (h->prof && h->nrec < kMaxRecords) {
        slot = h->nrec++;
        h->cls[slot] = cls;
        cudaEventRecord(h->ev[2 * slot], st);
    }
    const cudaError_t e = launch();
    if (slot >= 0) cudaEventRecord(h->ev[2 * slot + 1], st);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t esize(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

// Lazy calls read logits where they live: memory of the handle's device, or page-locked
// host memory that the device reaches at the same address (read over the host link).
// Anything else (another GPU's memory, pageable host memory, a registration mapped at
// another address) is refused.
// Whether p is host memory the device can read (pinned and mapped).
bool host_memory(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

bool readable_by_device(const void *p, int device) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == device;
    if (a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

int check_common(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                 const int32_t *tok, const int32_t *parent, const int32_t *accept_len,
                 const int32_t *out_tokens, const int32_t *kv_commit, const int32_t *bonus,
                 const int32_t *status) {
    if (!h) return SPEC_ERR_ARG;
    if (B < 0 || B > h->max_B) return SPEC_ERR_ARG;
    if (N < 1 || N > h->max_N || N > kMaxN) return SPEC_ERR_ARG;
    if (V < 1 || V > h->max_V) return SPEC_ERR_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    if (!logits || !tok || !parent || !accept_len || !out_tokens || !kv_commit || !bonus ||
        !status)
        return SPEC_ERR_ARG;
    if (!aligned(logits, esize(dtype))) return SPEC_ERR_ARG;
    const void *ints[] = {tok, parent, accept_len, out_tokens, kv_commit, bonus, status};
    for (const void *p : ints)
        if (!aligned(p, 4)) return SPEC_ERR_ARG;
    return SPEC_OK;
}

// Small batches: split every row over the most CTAs (8, 4 or 2) that still fit in one wave,
// so that the row-statistics kernel keeps every SM streaming. Only for row counts the
// workspace's per-piece arrays can hold.
void set_split(spec_handle h, RowStatsParams &rp) {
    rp.split = 1;
    if ((int64_t)rp.rows > (int64_t)h->max_B * h->max_N) return;
    rp.piece = h->piece;
    rp.count = h->count;
    for (int s = kRowChunks; s > 1; s /= 2)
        if ((int64_t)rp.rows * s <= h->slots) {
            rp.split = s;
            break;
        }
}

// Dense drafts, few requests: run each request's walk on a cluster of the most CTAs (8, 4 or
// 2) that still fit one wave of the walk kernel (one CTA per SM), so that its full-row passes
// over the target and draft rows are spread over that many SMs. Point drafts keep one CTA.
int walk_cluster(spec_handle h, int B, bool point) {
    if (point) return 1;
    const int64_t wave = h->sms;
    for (int c = 8; c > 1; c /= 2)
        if ((int64_t)B * c <= wave) return c;
    return 1;
}

// Debug builds, before a verify call's kernels: zero the request's violation words and every
// split-row arrival counter (so a counter an earlier call left wrong cannot spill over), then
// apply an injection armed by spec_debug_inject_arrival. Release builds do nothing.
int debug_prologue(spec_handle h, int B, int rows, cudaStream_t st) {
#ifdef SPEC_DEBUG
    const int64_t cap = (int64_t)h->max_B * h->max_N;
    if (cudaMemsetAsync(h->dbg, 0, sizeof(int32_t) * (size_t)B, st) != cudaSuccess ||
        cudaMemsetAsync(h->count, 0, sizeof(int32_t) * (size_t)cap, st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (h->inject_row >= 0 && h->inject_row < rows && h->inject_row < cap) {
        if (cudaMemcpyAsync(h->count + h->inject_row, &h->inject_value, sizeof(int32_t),
                            cudaMemcpyHostToDevice, st) != cudaSuccess)
            return SPEC_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
        h->inject_row = -1;
    }
#else
    (void)h;
    (void)B;
    (void)rows;
    (void)st;
#endif
    return SPEC_OK;
}

WalkOutputs outputs(int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                    int32_t *bonus, int32_t *status) {
    WalkOutputs o;
    o.accept_len = accept_len;
    o.out_tokens = out_tokens;
    o.kv_commit = kv_commit;
    o.bonus = bonus;
    o.status = status;
    return o;
}

int greedy_impl(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                const int32_t *tok, const int32_t *parent, WalkOutputs out, cudaStream_t st) {
    const int drc = debug_prologue(h, B, B * N, st);
    if (drc != SPEC_OK) return drc;
    RowStatsParams rp{};
    rp.x = logits;
    rp.V = V;
    rp.rows = B * N;
    rp.N = N;
    rp.k = 0.f;
    rp.m = h->m;
    rp.s = nullptr;
    rp.arg = h->arg;
    rp.flags = h->flags;
    rp.n_active = h->n_active;
    rp.dbg = h->dbg;
    set_split(h, rp);
    int rc = timed(h, SPEC_K_ROW_STATS, st,
                   [&] { return launch_row_stats(rp, dtype, ROW_GREEDY, st); });
    if (rc != SPEC_OK) return rc;
    GreedyWalkParams gp;
    gp.B = B;
    gp.N = N;
    gp.V = V;
    gp.parent = parent;
    gp.tok = tok;
    gp.arg = h->arg;
    gp.flags = h->flags;
    gp.out = out;
    gp.n_active = h->n_active;
    gp.dbg = h->dbg;
    return timed(h, SPEC_K_WALK_GREEDY, st, [&] { return launch_walk_greedy(gp, st); });
}

}  // namespace

extern "C" {

const char *spec_error_string(int code) {
    switch (code) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_ARG: return "invalid argument or outside the handle's limits";
        case SPEC_ERR_UNSUPPORTED: return "unsupported request";
        case SPEC_ERR_CUDA: return "CUDA call or kernel launch failed";
        case SPEC_ERR_WORKSPACE: return "workspace allocation failed";
        default: return "unknown error code";
    }
}

int spec_verify_init(spec_handle *out, int max_B, int max_N, int64_t max_V, int device) {
    SPEC_RANGE("spec_verify_init");
    if (!out) return SPEC_ERR_ARG;
    *out = nullptr;
    if (max_B < 1 || max_N < 1 || max_V < 1) return SPEC_ERR_ARG;
    if (max_N > kMaxN || max_V > kMaxV) return SPEC_ERR_UNSUPPORTED;
    if ((int64_t)max_B * max_N > (int64_t(1) << 30)) return SPEC_ERR_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return SPEC_ERR_CUDA;
    DeviceScope ds(device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    spec_ctx *h = new (std::nothrow) spec_ctx();
    if (!h) return SPEC_ERR_WORKSPACE;
    h->device = device;
    h->max_B = max_B;
    h->max_N = max_N;
    h->max_V = max_V;
    const size_t rows = (size_t)max_B * max_N;
    const size_t bytes =
        rows * (9 * 4 + kRowChunks * sizeof(float2) + kRowChunks * sizeof(RowPart) + 4) +
        sizeof(int32_t) * (size_t)max_B;
    if (cudaMalloc(&h->ws, bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return SPEC_ERR_WORKSPACE;
    }
    char *p = static_cast<char *>(h->ws);   // cudaMalloc: 256-byte aligned
    auto take = [&](size_t n) {
        char *q = p;
        p += n;
        return q;
    };
    h->chunk = reinterpret_cast<float2 *>(take(rows * kRowChunks * sizeof(float2)));
    h->piece = reinterpret_cast<RowPart *>(take(rows * kRowChunks * sizeof(RowPart)));
    h->m = reinterpret_cast<float *>(take(rows * 4));
    h->s = reinterpret_cast<float *>(take(rows * 4));
    h->pc = reinterpret_cast<float *>(take(rows * 4));
    h->mq = reinterpret_cast<float *>(take(rows * 4));
    h->sq = reinterpret_cast<float *>(take(rows * 4));
    h->qc = reinterpret_cast<float *>(take(rows * 4));
    h->arg = reinterpret_cast<int32_t *>(take(rows * 4));
    h->flags = reinterpret_cast<int32_t *>(take(rows * 4));
    h->dflags = reinterpret_cast<int32_t *>(take(rows * 4));
    h->count = reinterpret_cast<int32_t *>(take(rows * 4));
    h->dbg = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)max_B));
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaMemset(h->count, 0, rows * 4) != cudaSuccess ||
        cudaMemset(h->dbg, 0, sizeof(int32_t) * (size_t)max_B) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->ws);
        delete h;
        return SPEC_ERR_CUDA;
    }
    h->slots = kSplitCtasPerSm * sms;   // one wave of the split row-statistics kernel
    h->sms = sms;
    *out = h;
    return SPEC_OK;
}

int spec_verify_destroy(spec_handle h) {
    SPEC_RANGE("spec_verify_destroy");
    if (!h) return SPEC_OK;
    DeviceScope ds(h->device);
    if (h->ev_ready)
        for (int i = 0; i < 2 * kMaxRecords; ++i) cudaEventDestroy(h->ev[i]);
    cudaFree(h->ws);
    delete h;
    return SPEC_OK;
}

int spec_build_tree_mask(spec_handle h, const int32_t *parent, int B, int N, uint64_t *anc_mask,
                         int32_t *depth, int32_t *status, void *stream) {
    SPEC_RANGE("spec_build_tree_mask");
    if (!h) return SPEC_ERR_ARG;
    if (B < 0 || B > h->max_B || N < 1 || N > h->max_N || N > kMaxN) return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    if (!parent || !anc_mask || !depth || !status) return SPEC_ERR_ARG;
    if (!aligned(parent, 4) || !aligned(anc_mask, 8) || !aligned(depth, 4) || !aligned(status, 4))
        return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return timed(h, SPEC_K_TREE_MASK, st, [&] {
        return launch_tree_mask(parent, B, N, anc_mask, depth, status, st);
    });
}

int spec_verify_greedy(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                       const int32_t *draft_token, const int32_t *parent, int32_t *accept_len,
                       int32_t *out_tokens, int32_t *kv_commit, int32_t *bonus, int32_t *status,
                       void *stream) {
    SPEC_RANGE("spec_verify_greedy");
    int rc = check_common(h, logits, dtype, B, N, V, draft_token, parent, accept_len,
                          out_tokens, kv_commit, bonus, status);
    if (rc != SPEC_OK || B == 0) return rc;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    return greedy_impl(h, logits, dtype, B, N, V, draft_token, parent,
                       outputs(accept_len, out_tokens, kv_commit, bonus, status),
                       static_cast<cudaStream_t>(stream));
}

int spec_verify_sample(spec_handle h, const void *logits, int dtype, int B, int N, int64_t V,
                       const int32_t *draft_token, const int32_t *parent, const void *draft,
                       int draft_kind, int draft_dtype, float temperature,
                       const float *uniforms, int32_t *accept_len, int32_t *out_tokens,
                       int32_t *kv_commit, int32_t *bonus, int32_t *status, void *stream) {
    SPEC_RANGE("spec_verify_sample");
    int rc = check_common(h, logits, dtype, B, N, V, draft_token, parent, accept_len,
                          out_tokens, kv_commit, bonus, status);
    if (rc != SPEC_OK) return rc;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return SPEC_ERR_ARG;
    const float k = temperature > 0.f ? kLog2eF / temperature : 0.f;
    if (temperature > 0.f && !std::isfinite(k)) return SPEC_ERR_ARG;
    if (draft_kind != SPEC_DRAFT_POINT && draft_kind != SPEC_DRAFT_PROBS_F32 &&
        draft_kind != SPEC_DRAFT_LOGITS)
        return SPEC_ERR_ARG;
    if (draft_kind == SPEC_DRAFT_LOGITS && draft_dtype != SPEC_F32 && draft_dtype != SPEC_BF16)
        return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WalkOutputs out = outputs(accept_len, out_tokens, kv_commit, bonus, status);
    if (temperature == 0.f)
        return greedy_impl(h, logits, dtype, B, N, V, draft_token, parent, out, st);
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_ARG;
    const bool dense = draft_kind != SPEC_DRAFT_POINT;
    if (dense) {
        if (!draft) return SPEC_ERR_ARG;
        const size_t de = draft_kind == SPEC_DRAFT_LOGITS ? esize(draft_dtype) : 4;
        if (!aligned(draft, de)) return SPEC_ERR_ARG;
    }
    rc = debug_prologue(h, B, B * N, st);
    if (rc != SPEC_OK) return rc;

    RowStatsParams rp{};
    rp.x = logits;
    rp.V = V;
    rp.rows = B * N;
    rp.N = N;
    rp.k = k;
    rp.parent = parent;
    rp.tok = draft_token;
    rp.skip_leaves = 0;
    rp.pc_normalized = 0;
    rp.m = h->m;
    rp.s = h->s;
    rp.arg = nullptr;
    rp.flags = h->flags;
    rp.pc = h->pc;
    rp.n_active = h->n_active;
    rp.chunk = h->chunk;
    rp.dbg = h->dbg;
    if (!dense) {
        set_split(h, rp);
        rc = timed(h, SPEC_K_ROW_STATS, st,
                   [&] { return launch_row_stats(rp, dtype, ROW_SAMPLE, st); });
        if (rc != SPEC_OK) return rc;
    } else {
        // The draft rows of the inner nodes are streamed in the same launch as the target rows.
        RowStatsParams dp = rp;
        dp.x = draft;
        dp.chunk = nullptr;   // partials are kept for the target rows only
        dp.skip_leaves = 1;
        dp.flags = h->dflags;
        dp.pc = h->qc;
        int mode = ROW_PROBS, ddt = SPEC_F32;
        if (draft_kind == SPEC_DRAFT_LOGITS) {
            mode = ROW_SAMPLE;
            ddt = draft_dtype;
            dp.m = h->mq;
            dp.s = h->sq;
        } else {
            dp.m = nullptr;
            dp.s = nullptr;
        }
        rc = timed(h, SPEC_K_ROW_STATS, st, [&] {
            return launch_row_stats_pair(rp, dtype, dp, ddt, mode, st);
        });
        if (rc != SPEC_OK) return rc;
    }

    SampleWalkParams wp{};
    wp.B = B;
    wp.N = N;
    wp.V = V;
    wp.dtype = dtype;
    wp.logits = logits;
    wp.parent = parent;
    wp.tok = draft_token;
    wp.uniforms = uniforms;
    wp.k = k;
    wp.m = h->m;
    wp.s = h->s;
    wp.pc = h->pc;
    wp.flags = h->flags;
    wp.draft_kind = draft_kind;
    wp.draft_dtype = draft_dtype;
    wp.draft = draft;
    wp.mq = h->mq;
    wp.sq = h->sq;
    wp.qc = h->qc;
    wp.dflags = h->dflags;
    wp.out = out;
    wp.n_active = h->n_active;
    wp.chunk = draft_kind == SPEC_DRAFT_POINT ? h->chunk : nullptr;
    wp.cluster = walk_cluster(h, B, draft_kind == SPEC_DRAFT_POINT);
    wp.dbg = h->dbg;
    return timed(h, SPEC_K_WALK_SAMPLE, st, [&] { return launch_walk_sample(wp, st); });
}

int spec_verify_greedy_lazy(spec_handle h, const void *logits, int dtype, int B, int N,
                            int64_t V, const int32_t *draft_token, const int32_t *parent,
                            int32_t *accept_len, int32_t *out_tokens, int32_t *kv_commit,
                            int32_t *bonus, int32_t *status, void *stream) {
    SPEC_RANGE("spec_verify_greedy_lazy");
    int rc = check_common(h, logits, dtype, B, N, V, draft_token, parent, accept_len,
                          out_tokens, kv_commit, bonus, status);
    if (rc != SPEC_OK || B == 0) return rc;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    if (!readable_by_device(logits, h->device)) return SPEC_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = debug_prologue(h, B, 0, st);
    if (rc != SPEC_OK) return rc;
    LazyGreedyParams lp;
    lp.B = B;
    lp.N = N;
    lp.V = V;
    lp.dtype = dtype;
    lp.logits = logits;
    lp.parent = parent;
    lp.tok = draft_token;
    lp.out = outputs(accept_len, out_tokens, kv_commit, bonus, status);
    lp.n_active = h->n_active;
    lp.dbg = h->dbg;
    return timed(h, SPEC_K_LAZY_GREEDY, st, [&] { return launch_lazy_greedy(lp, st); });
}

int spec_verify_sample_lazy(spec_handle h, const void *logits, int dtype, int B, int N,
                            int64_t V, const int32_t *draft_token, const int32_t *parent,
                            const void *draft, int draft_kind, int draft_dtype, float temperature,
                            const float *uniforms, int32_t *accept_len, int32_t *out_tokens,
                            int32_t *kv_commit, int32_t *bonus, int32_t *status, void *stream) {
    SPEC_RANGE("spec_verify_sample_lazy");
    int rc = check_common(h, logits, dtype, B, N, V, draft_token, parent, accept_len,
                          out_tokens, kv_commit, bonus, status);
    if (rc != SPEC_OK) return rc;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return SPEC_ERR_ARG;
    const float k = temperature > 0.f ? kLog2eF / temperature : 0.f;
    if (temperature > 0.f && !std::isfinite(k)) return SPEC_ERR_ARG;
    if (draft_kind != SPEC_DRAFT_POINT && draft_kind != SPEC_DRAFT_PROBS_F32 &&
        draft_kind != SPEC_DRAFT_LOGITS)
        return SPEC_ERR_ARG;
    if (draft_kind == SPEC_DRAFT_LOGITS && draft_dtype != SPEC_F32 && draft_dtype != SPEC_BF16)
        return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    if (temperature == 0.f)
        return spec_verify_greedy_lazy(h, logits, dtype, B, N, V, draft_token, parent,
                                       accept_len, out_tokens, kv_commit, bonus, status, stream);
    if (!uniforms || !aligned(uniforms, 4)) return SPEC_ERR_ARG;
    if (draft_kind != SPEC_DRAFT_POINT) {
        if (!draft) return SPEC_ERR_ARG;
        const size_t de = draft_kind == SPEC_DRAFT_LOGITS ? esize(draft_dtype) : 4;
        if (!aligned(draft, de)) return SPEC_ERR_ARG;
    }
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    if (!readable_by_device(logits, h->device) ||
        (draft && !readable_by_device(draft, h->device)))
        return SPEC_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = debug_prologue(h, B, 0, st);
    if (rc != SPEC_OK) return rc;
    SampleWalkParams wp{};
    wp.B = B;
    wp.N = N;
    wp.V = V;
    wp.dtype = dtype;
    wp.logits = logits;
    wp.parent = parent;
    wp.tok = draft_token;
    wp.uniforms = uniforms;
    wp.k = k;
    wp.draft_kind = draft_kind;
    wp.draft_dtype = draft_dtype;
    wp.draft = draft;
    wp.lazy = 1;
    wp.host_rows = host_memory(logits);
    wp.out = outputs(accept_len, out_tokens, kv_commit, bonus, status);
    wp.n_active = h->n_active;
    wp.dbg = h->dbg;
    return timed(h, SPEC_K_LAZY_SAMPLE, st, [&] { return launch_walk_sample(wp, st); });
}

int spec_set_node_budget(spec_handle h, const int32_t *n_active) {
    SPEC_RANGE("spec_set_node_budget");
    if (!h) return SPEC_ERR_ARG;
    if (n_active && !aligned(n_active, 4)) return SPEC_ERR_ARG;
    h->n_active = n_active;
    return SPEC_OK;
}

int spec_budget_update(spec_handle h, const spec_budget_params *params,
                       const int32_t *accept_len, const int32_t *status, const int32_t *parent,
                       int B, int N, spec_budget_state *state, int32_t *n_active, void *stream) {
    SPEC_RANGE("spec_budget_update");
    if (!h || !params || !state || !n_active) return SPEC_ERR_ARG;
    if (B < 0 || B > h->max_B || N < 1 || N > h->max_N || N > kMaxN) return SPEC_ERR_ARG;
    const spec_budget_params &q = *params;
    if (!(q.target > 0.0 && q.target <= 1.0) || !(q.alpha > 0.0 && q.alpha <= 1.0) ||
        !(q.band >= 0.0) || !std::isfinite(q.band))
        return SPEC_ERR_ARG;
    if (q.n_min < 1 || q.n_min > q.n_max || q.n_max > N || q.step < 1) return SPEC_ERR_ARG;
    if (B > 0 && (!accept_len || !status || !parent)) return SPEC_ERR_ARG;
    const void *ints[] = {accept_len, status, parent, n_active};
    for (const void *p : ints)
        if (p && !aligned(p, 4)) return SPEC_ERR_ARG;
    if (!aligned(state, alignof(spec_budget_state))) return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BudgetParams bp;
    bp.prm = q;
    bp.accept_len = accept_len;
    bp.status = status;
    bp.parent = parent;
    bp.B = B;
    bp.N = N;
    bp.state = state;
    bp.n_active = n_active;
    return timed(h, SPEC_K_BUDGET, st, [&] { return launch_budget_update(bp, st); });
}

int spec_kv_commit(spec_handle h, const void *src_k, const void *src_v, int src_dtype, int B,
                   int N, int H, int D, const int32_t *kv_commit, const int32_t *accept_len,
                   void *cache_k, void *cache_v, int cache_kind, int layout, int block_size,
                   int64_t num_blocks, const int32_t *block_table, int max_blocks,
                   const int32_t *seq_pos, const float *k_scale, const float *v_scale,
                   int scale_per_token, int32_t *commit_status, void *stream) {
    SPEC_RANGE("spec_kv_commit");
    if (!h) return SPEC_ERR_ARG;
    if (B < 0 || B > h->max_B || N < 1 || N > h->max_N || N > kMaxN) return SPEC_ERR_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > (int64_t(1) << 24)) return SPEC_ERR_ARG;
    if (src_dtype != SPEC_F32 && src_dtype != SPEC_BF16 && src_dtype != SPEC_F16)
        return SPEC_ERR_ARG;
    if (cache_kind != SPEC_CACHE_SAME && cache_kind != SPEC_CACHE_FP8_E4M3 &&
        cache_kind != SPEC_CACHE_FP8_E5M2)
        return SPEC_ERR_ARG;
    if (layout != SPEC_KV_NHD && layout != SPEC_KV_HND) return SPEC_ERR_ARG;
    if (scale_per_token != SPEC_SCALE_TENSOR && scale_per_token != SPEC_SCALE_PER_TOKEN)
        return SPEC_ERR_ARG;
    if (block_size < 1 || num_blocks < 1 || num_blocks > INT32_MAX || max_blocks < 1)
        return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    if (!src_k || !src_v || !kv_commit || !accept_len || !cache_k || !cache_v || !block_table ||
        !seq_pos)
        return SPEC_ERR_ARG;
    const size_t se = src_dtype == SPEC_F32 ? 4 : 2;
    const size_t ce = cache_kind == SPEC_CACHE_SAME ? se : 1;
    if (!aligned(src_k, se) || !aligned(src_v, se) || !aligned(cache_k, ce) ||
        !aligned(cache_v, ce))
        return SPEC_ERR_ARG;
    const void *ints[] = {kv_commit, accept_len, block_table, seq_pos};
    for (const void *p : ints)
        if (!aligned(p, 4)) return SPEC_ERR_ARG;
    if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)) ||
        (commit_status && !aligned(commit_status, 4)))
        return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    KvCommitParams kp;
    kp.src_k = src_k;
    kp.src_v = src_v;
    kp.src_dtype = src_dtype;
    kp.B = B;
    kp.N = N;
    kp.H = H;
    kp.D = D;
    kp.kv_commit = kv_commit;
    kp.accept_len = accept_len;
    kp.cache_k = cache_k;
    kp.cache_v = cache_v;
    kp.cache_kind = cache_kind;
    kp.layout = layout;
    kp.block_size = block_size;
    kp.num_blocks = num_blocks;
    kp.block_table = block_table;
    kp.max_blocks = max_blocks;
    kp.seq_pos = seq_pos;
    kp.k_scale = k_scale;
    kp.v_scale = v_scale;
    kp.scale_per_token = scale_per_token;
    kp.status = commit_status;
    kp.sms = h->sms;
    // 8 elements per thread step: rows of D elements and 16-byte aligned bases.
    const bool vec = D % 8 == 0 && aligned(src_k, 16) && aligned(src_v, 16) &&
                     aligned(cache_k, 16) && aligned(cache_v, 16);
#ifdef SPEC_DEBUG
    // debug builds combine statuses with atomicMax, from zero
    if (commit_status &&
        cudaMemsetAsync(commit_status, 0, sizeof(int32_t) * (size_t)B, st) != cudaSuccess)
        return SPEC_ERR_CUDA;
#endif
    return timed(h, SPEC_K_KV_COMMIT, st, [&] { return launch_kv_commit(kp, vec, st); });
}

int spec_row_stats(spec_handle h, const void *logits, int dtype, int rows, int N, int64_t V,
                   float temperature, const int32_t *draft_token, const int32_t *parent,
                   float *row_max, float *row_sum, int32_t *row_argmax, int32_t *row_flags,
                   float *child_prob, void *stream) {
    SPEC_RANGE("spec_row_stats");
    if (!h) return SPEC_ERR_ARG;
    if (rows < 0 || N < 1 || N > kMaxN || V < 1 || V > kMaxV) return SPEC_ERR_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_ARG;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return SPEC_ERR_ARG;
    const float k = temperature > 0.f ? kLog2eF / temperature : 0.f;
    if (temperature > 0.f && !std::isfinite(k)) return SPEC_ERR_ARG;
    const bool gather = draft_token && parent && child_prob;
    if (gather && (temperature == 0.f || rows % N != 0)) return SPEC_ERR_ARG;
    if (rows == 0) return SPEC_OK;
    if (!logits || !row_max || !row_sum || !row_argmax || !row_flags) return SPEC_ERR_ARG;
    if (!aligned(logits, esize(dtype))) return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    RowStatsParams rp{};
    rp.x = logits;
    rp.V = V;
    rp.rows = rows;
    rp.N = N;
    rp.k = k;
    rp.parent = gather ? parent : nullptr;
    rp.tok = gather ? draft_token : nullptr;
    rp.skip_leaves = 0;
    rp.pc_normalized = 1;
    rp.m = row_max;
    rp.s = row_sum;
    rp.arg = row_argmax;
    rp.flags = row_flags;
    rp.pc = gather ? child_prob : nullptr;
    set_split(h, rp);
    if (rp.split > 1) {
        const int drc = debug_prologue(h, 0, rows, st);
        if (drc != SPEC_OK) return drc;
    }
    const int mode = temperature > 0.f ? ROW_SAMPLE : ROW_GREEDY;
    return timed(h, SPEC_K_ROW_STATS, st, [&] { return launch_row_stats(rp, dtype, mode, st); });
}

int spec_profile_begin(spec_handle h) {
    if (!h) return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    if (!h->ev_ready) {
        for (int i = 0; i < 2 * kMaxRecords; ++i)
            if (cudaEventCreate(&h->ev[i]) != cudaSuccess) return SPEC_ERR_CUDA;
        h->ev_ready = true;
    }
    h->nrec = 0;
    h->prof = true;
    return SPEC_OK;
}

int spec_profile_end(spec_handle h, float *ms_per_class, int32_t *launches_per_class) {
    if (!h || !ms_per_class || !launches_per_class) return SPEC_ERR_ARG;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    for (int c = 0; c < SPEC_K_COUNT; ++c) {
        ms_per_class[c] = 0.f;
        launches_per_class[c] = 0;
    }
    int rc = SPEC_OK;
    for (int i = 0; i < h->nrec; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(h->ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]) != cudaSuccess) {
            rc = SPEC_ERR_CUDA;
            continue;
        }
        ms_per_class[h->cls[i]] += ms;
        launches_per_class[h->cls[i]] += 1;
    }
    h->prof = false;
    h->nrec = 0;
    return rc;
}

int spec_debug_build(void) {
    SPEC_RANGE("spec_debug_build");
#ifdef SPEC_DEBUG
    return 1;
#else
    return 0;
#endif
}

int spec_debug_inject_arrival(spec_handle h, int row, int value) {
    SPEC_RANGE("spec_debug_inject_arrival");
#ifdef SPEC_DEBUG
    if (!h || row < 0 || (int64_t)row >= (int64_t)h->max_B * h->max_N) return SPEC_ERR_ARG;
    h->inject_row = row;
    h->inject_value = value;
    return SPEC_OK;
#else
    (void)h;
    (void)row;
    (void)value;
    return SPEC_ERR_UNSUPPORTED;
#endif
}

int spec_debug_words(spec_handle h, int32_t *words, int B, void *stream) {
    SPEC_RANGE("spec_debug_words");
#ifdef SPEC_DEBUG
    if (!h || B < 0 || B > h->max_B || (B > 0 && !words)) return SPEC_ERR_ARG;
    if (B == 0) return SPEC_OK;
    DeviceScope ds(h->device);
    if (!ds.ok()) return SPEC_ERR_CUDA;
    return cudaMemcpyAsync(words, h->dbg, sizeof(int32_t) * (size_t)B, cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
#else
    (void)h;
    (void)words;
    (void)B;
    (void)stream;
    return SPEC_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
