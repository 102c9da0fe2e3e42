// Sampling tree walk, inverse-CDF bonus draw and accepted-path compaction (kernel templates;
// instantiated by walk_sample_point.cu and walk_sample_dense.cu).
//
// EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput",
// commit 4b728e2: sampling uses standard (SpecInfer-style) rejection sampling against the
// draft, so the output distribution is the target's. From the root the walk tests the
// children of the current node in ascending node index; an accepted child becomes the
// current node; when no child is accepted (or the node is a leaf) a bonus token is drawn
// from the residual distribution by inverse CDF with the request's last uniform.
//
// One CTA of 512 threads per request. Warp 0 runs the walk on scalars gathered by the
// row-statistics kernel (e_t = 2^((z_t - m) log2(e)/T) at every child token, the row sums S,
// and the same for dense draft rows); the children of a node are one 64-bit ballot mask.
// Whenever a decision needs a sum over the vocabulary, all 16 warps stream the node's row
// once ("pass"):
//   * point drafts: p(t) / sum_{v not in R} p(v) is formed as e_t / (S - sum_{v in R} e_v);
//     when the rejected mass exceeds 15/16 of the denominator the remainder is re-summed;
//   * dense drafts: after a rejection with siblings left, Z = sum_v max(r(v) - q(v), 0)
//     normalises the next residual level;
//   * bonus: the residual at the stop node is summed per 256-element sub-tile (a warp scan
//     over 32 lanes x 8 elements), the sub-tile sums stay in shared memory, warp 0 locates
//     the sub-tile holding tau = u * S (scan of per-lane groups of sub-tile sums, then of the
//     chosen group) and re-reads only that sub-tile to find the token. With point drafts the
//     pass covers one chunk of the row only: the row-statistics kernel (eager) or the lazy
//     pass leaves the (max, sum) of every chunk of the row, from which warp 0 first picks the
//     chunk holding tau (the rejected tokens' mass taken out of their chunks).
// Every search level falls back to the last token with r(v) > 0 when rounding leaves tau past
// its end, so the drawn token always has positive residual mass.
// Lazy walks (no row-statistics kernel) stream each row they visit when they enter it, one
// chunk per warp with the row-statistics kernel's per-element code.
// A pass issues the 16-byte loads of 8 sub-tiles per lane before using any of them (2 CTAs
// per SM: 128 KiB of each SM's loads in flight); sums use compensated float32, and the
// float64 pipe (slow on this part) only sees a handful of operations per decision.

#pragma once

#include <climits>

#include "row_pass.cuh"
#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

// Sub-tiles in flight per warp in a dense-draft pass: 4 when the target and draft rows are
// both 16-bit (8 KiB of loads in flight per warp), 2 when either is f32 (4 in flight spilled
// there).
#ifndef SPEC_DENSE_PASS_UNROLL
#define SPEC_DENSE_PASS_UNROLL 4
#endif
// 16-byte loads in flight per thread in the lazy row pass's register loop: rows in host memory
// (read over the host link: 0.403 ms per large-tree call with 4, 0.413 ms with 2) and rows that
// are not 16-byte aligned.
#ifndef SPEC_LAZY_UNROLL
#define SPEC_LAZY_UNROLL 4
#endif
// Lazy row passes over 16-byte aligned rows stage their loads through a ring of cp.async
// copies in shared memory instead: SPEC_LAZY_RING vectors in flight per thread (32 KiB per
// CTA), twice the register loads, without holding registers. Measured on the large tree (lazy
// sampling call): 45.5 us without the ring, 34.9 us with 4 or 6 slots, 35.3 us with 10; at
// mean accept length 1.41, 120 / 99.9 / 100.8 / 107 us.
#ifndef SPEC_LAZY_RING
#define SPEC_LAZY_RING 4
#endif

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSub = kSubTile;   // elements per sub-tile: 32 lanes x 8

// Point-draft bonus draws within one row chunk (chunk_draw): each warp holds up to
// draw_subs sub-tiles of the chunk in registers.
template <int DT>
constexpr int draw_subs() { return DT == 1 ? 8 : 4; }
// Floats of the sub-tile sums in dynamic shared memory.
__host__ __device__ __forceinline__ int subsum_floats(int64_t V) {
    return (int)((V + kSub - 1) / kSub);
}
// Lazy walks: the cp.async ring follows the sub-tile sums, 16-byte aligned.
__host__ __device__ __forceinline__ int lazy_ring_offset(int64_t V) {
    return (subsum_floats(V) + 3) & ~3;
}
constexpr size_t kLazyRingBytes = (size_t)kThreads * SPEC_LAZY_RING * 16;

enum { CMD_NONE = 0, CMD_DONE, CMD_BONUS, CMD_PASS_SR, CMD_PASS_Z, CMD_STATS };

// 16-byte asynchronous copy global -> shared (bypassing L1), one commit group per call site,
// and the wait until at most N of this thread's groups are still in flight (a hardware wait on
// the thread's own copies: nothing spins).
__device__ __forceinline__ void cp_async16(uint4 *smem, const uint4 *gmem) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct Smem {
    int par[kMaxN], tok[kMaxN], flags[kMaxN], dflags[kMaxN];
    float ec[kMaxN];     // e_t of each child in its parent's target row
    float eqc[kMaxN];    // draft: e_q at each child token (probabilities: q itself)
    float s[kMaxN], m[kMaxN], sq[kMaxN], mq[kMaxN];
    float u[kMaxN + 1];
    int path[kMaxN];
    int R[kMaxN];        // rejected tokens at the current node, ascending
    float RE[kMaxN];     // e_t of each rejected token (same order as R)
    float invZ[kMaxN];   // dense: 1 / Z of each normalised residual level (0: level kept)
    double zinv[kMaxN];  // dense: 1 / Z of each level in float64 (0: level kept)
    int nR, nlev, pending;
    int cmd, node, L, st, bonus;
    double total;
    double wtot[kWarps];
    int haskids;                       // lazy statistics: the node has children
    int cpick;                         // eager point bonus: chosen row chunk (-1: none)
    double ctau;                       // ... and tau relative to the chunk's start
    unsigned cmask;                    // eager point re-sum: chunks summed exactly (bit = chunk)
    double ckeep;                      // ... mass of the other chunks, from their partials
    int cpart_node;                    // lazy: node whose chunk partials are in cpart[]
    float2 cpart[kLazyChunks];         // lazy: (max, sum) of each chunk of that node's row
    float2 epart[kMaxN][kRowChunks];   // eager point drafts: chunk partials of every node's row
    int wflag[kWarps];
    rowpass::Part part[kWarps], part_out;
    double ctot;   // clusters: this CTA's share of a pass total
    int bcast;     // clusters: a control value of the leading CTA
    int dbgv;      // debug builds: violation bits found by this CTA
    float dtot[kWarps];      // chunk draw: each warp's block total
    float dsub[kWarps][8];   // ... and its sub-tile totals
};

// Debug builds: record a violation found while walking request (CTA) state in shared memory;
// it is charged to the request when the walk ends. Returns `ok` (always true in release).
__device__ __forceinline__ bool walk_check(bool ok, Smem &sm, int bit) {
    if constexpr (kDebug) {
        if (!ok) atomicOr(&sm.dbgv, bit);
        return ok;
    } else {
        return true;
    }
}

// Clusters (CL CTAs per request): every CTA runs the same walk on the same data, but each
// branch that is followed by a cluster barrier takes the leading CTA's value, so all CTAs
// pass the same barriers even if their own values differed. `v` is block-uniform.
template <int CL>
__device__ __forceinline__ int lead(Smem &sm, int v) {
    if constexpr (CL == 1) {
        return v;
    } else {
        if (threadIdx.x == 0) sm.bcast = v;
        cluster_sync();
        const int r = ld_cluster_s32(cluster_addr(&sm.bcast, 0));
        cluster_sync();
        return r;
    }
}

struct Ctx {
    const char *zrow;    // target row of the node
    const char *drow;    // draft row of the node (dense drafts)
    float negm, invS, negmq, invSq, k;
    int V;
    bool zvec, dvec;     // rows 16-byte aligned
    bool useq;           // dense residual levels present: the draft row is read
};

// ---- element access -------------------------------------------------------------------------

template <int DT>
__device__ __forceinline__ void fetch(const char *row, int e0, uint4 &a, uint4 &b) {
    if (DT == 1) {
        a = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 8);
    } else {
        a = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4);
        b = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4 + 1);
    }
}

// fetch, skipping the vectors that start at or past `lim` (they read as zeros).
template <int DT>
__device__ __forceinline__ void fetch_below(const char *row, int e0, int lim, uint4 &a, uint4 &b) {
    a = b = make_uint4(0u, 0u, 0u, 0u);
    if (DT == 1) {
        if (e0 < lim) a = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 8);
    } else {
        if (e0 < lim) a = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4);
        if (e0 + 4 < lim) b = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4 + 1);
    }
}

// No mass for the elements e0 + q at or past V.
__device__ __forceinline__ void mask_past(float (&r)[8], int e0, int V) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (e0 + q >= V) r[q] = 0.f;
}

// x[q] = value(e0 + q) + c for 8 elements held in one (bf16) or two (f32) 16-byte vectors.
template <int DT>
__device__ __forceinline__ void shifted8(const uint4 &a, const uint4 &b, float c, float (&x)[8]) {
    if (DT == 1) {
        bf_add2(a.x, c, x[0], x[1]);
        bf_add2(a.y, c, x[2], x[3]);
        bf_add2(a.z, c, x[4], x[5]);
        bf_add2(a.w, c, x[6], x[7]);
    } else {
        x[0] = __uint_as_float(a.x) + c; x[1] = __uint_as_float(a.y) + c;
        x[2] = __uint_as_float(a.z) + c; x[3] = __uint_as_float(a.w) + c;
        x[4] = __uint_as_float(b.x) + c; x[5] = __uint_as_float(b.y) + c;
        x[6] = __uint_as_float(b.z) + c; x[7] = __uint_as_float(b.w) + c;
    }
}

// The same with scalar loads; positions at or beyond V read as `fill` (before the shift).
template <int DT>
__device__ __forceinline__ void shifted8_scalar(const char *row, int e0, int V, float c,
                                                float fill, float (&x)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = (e0 + q < V ? load_elem<DT>(row, e0 + q) : fill) + c;
}

// Residual r(v) of 8 elements from the shifted target values zs = z - m and, for dense drafts,
// the shifted draft values ds = d - m_q (logits) or the draft probabilities (PROBS_F32).
template <int DK>
__device__ __forceinline__ void residual8(const Ctx &c, const Smem &sm, const float (&zs)[8],
                                          const float (&ds)[8], float (&r)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float e = ex2(zs[q] * c.k);
        if (DK == DRAFT_POINT) {
            r[q] = e;
        } else {
            float x = e * c.invS;
            if (c.useq) {
                const float qv = DK == DRAFT_LOGITS ? ex2(ds[q] * c.k) * c.invSq : ds[q];
                for (int l = 0; l < sm.nlev; ++l)
                    if (sm.invZ[l] > 0.f) x = fmaxf(x - qv, 0.f) * sm.invZ[l];
                if (sm.pending) x = fmaxf(x - qv, 0.f);
            }
            r[q] = x;
        }
    }
}

// Point drafts: zero the rejected tokens inside sub-tile j. `rc` is a warp-uniform cursor
// into the ascending rejected list (sub-tiles of one warp are visited in increasing order).
__device__ __forceinline__ void zero_rejected(const Smem &sm, int j, int lane, int &rc,
                                              float (&r)[8]) {
    const int lo = j * kSub, hi = lo + kSub;
    const int nR = sm.nR;
    while (rc < nR && sm.R[rc] < lo) ++rc;
    if (rc < nR && sm.R[rc] < hi) {
        const int e0 = lo + lane * 8;
        for (int i = rc; i < nR && sm.R[i] < hi; ++i) {
            const int t = sm.R[i] - e0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (t == q) r[q] = 0.f;
        }
    }
}

// Residual of the 8 elements of sub-tile j owned by this lane, with every check needed when
// the sub-tile may be ragged or the rows unaligned.
template <int DT, int DK, int DDT>
__device__ __forceinline__ void residual8_any(const Ctx &c, const Smem &sm, int j, int lane,
                                              int &rc, float (&r)[8]) {
    constexpr int kDDT = DK == DRAFT_LOGITS ? DDT : 0;
    const int e0 = j * kSub + lane * 8;
    float zs[8], ds[8];
    const bool vec = c.zvec && (DK == DRAFT_POINT || !c.useq || c.dvec) && e0 + 8 <= c.V;
    if (vec) {
        uint4 za, zb, da, db;
        fetch<DT>(c.zrow, e0, za, zb);
        if (DK != DRAFT_POINT && c.useq) fetch<kDDT>(c.drow, e0, da, db);
        shifted8<DT>(za, zb, c.negm, zs);
        if (DK == DRAFT_LOGITS && c.useq) shifted8<kDDT>(da, db, c.negmq, ds);
        if (DK == DRAFT_PROBS_F32 && c.useq) shifted8<0>(da, db, 0.f, ds);
    } else {
        shifted8_scalar<DT>(c.zrow, e0, c.V, c.negm, -INFINITY, zs);
        if (DK == DRAFT_LOGITS && c.useq)
            shifted8_scalar<kDDT>(c.drow, e0, c.V, c.negmq, -INFINITY, ds);
        if (DK == DRAFT_PROBS_F32 && c.useq) shifted8_scalar<0>(c.drow, e0, c.V, 0.f, 0.f, ds);
    }
    residual8<DK>(c, sm, zs, ds, r);
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (e0 + q >= c.V) r[q] = 0.f;
    if (DK == DRAFT_POINT) zero_rejected(sm, j, lane, rc, r);
}

// Compensated (Kahan) float accumulation: the error stays near one float rounding however
// many terms are added, without the slow float64 pipe.
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ double value() const { return (double)s - (double)c; }
};

__device__ __forceinline__ float sum8(const float (&r)[8]) {
    float ls = r[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) ls += r[q];
    return ls;
}

// ---- one pass over the node's residual ----------------------------------------------------

// Every warp sums its sub-tiles of [jlo, jhi) (default: the whole row) into subsum[] (one warp
// scan per 256 elements); with `total`, their sum lands in sm.total. All threads call it; it
// ends synchronised. With clusters (CL > 1) the CL * 16 warps of the cluster share the
// sub-tiles (warp w of CTA r takes those with (j - jlo) mod 16 CL = 16 r + w); afterwards every
// CTA holds all of the range's sub-tile sums and the same total (CTA shares added in rank
// order).
template <int DT, int DK, int DDT, int CL = 1>
__device__ void residual_pass(const Ctx &c, Smem &sm, float *subsum, int jlo = 0,
                              int jhi = INT_MAX, bool total = true) {
    // sub-tiles in flight per warp (32 registers of raw loads)
    constexpr int U = DK == DRAFT_POINT                          ? (DT == 1 ? 8 : 4)
                      : DT == 1 && DK == DRAFT_LOGITS && DDT == 1 ? SPEC_DENSE_PASS_UNROLL
                                                                  : 2;
    constexpr int kDDT = DK == DRAFT_LOGITS ? DDT : 0;
    constexpr int GW = CL * kWarps;   // warps sharing the pass
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = CL == 1 ? 0 : cluster_rank();
    const int gw = rank * kWarps + warp;
    const int nsub = min((c.V + kSub - 1) / kSub, jhi);
    const bool vec = c.zvec && (DK == DRAFT_POINT || !c.useq || c.dvec);
    const int nfull = min(vec ? c.V / kSub : 0, nsub);
    KSum wsum;
    int rc = 0;

    for (int j0 = jlo + gw; j0 < nfull; j0 += GW * U) {
        uint4 za[U], zb[U], da[U], db[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * GW;
            if (j < nfull) {
                const int e0 = j * kSub + lane * 8;
                fetch<DT>(c.zrow, e0, za[u], zb[u]);
                if (DK != DRAFT_POINT && c.useq) fetch<kDDT>(c.drow, e0, da[u], db[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * GW;
            if (j < nfull) {
                float zs[8], ds[8], r[8];
                shifted8<DT>(za[u], zb[u], c.negm, zs);
                if (DK == DRAFT_LOGITS && c.useq) shifted8<kDDT>(da[u], db[u], c.negmq, ds);
                if (DK == DRAFT_PROBS_F32 && c.useq) shifted8<0>(da[u], db[u], 0.f, ds);
                residual8<DK>(c, sm, zs, ds, r);
                if (DK == DRAFT_POINT) zero_rejected(sm, j, lane, rc, r);
                const float incl = warp_incl_scan(sum8(r));
                if (lane == 31 && walk_check(j < (c.V + kSub - 1) / kSub, sm, DBG_INDEX)) {
                    subsum[j] = incl;
                    wsum.add(incl);
                }
            }
        }
    }
    // Ragged last sub-tile, or every sub-tile of a row that is not 16-byte aligned.
    int j1 = max(nfull, jlo) + warp;
    if (CL > 1) {   // keep the cluster's assignment of sub-tiles to warps
        j1 = jlo + gw;
        const int start = max(nfull, jlo);
        if (j1 < start) j1 += (start - j1 + GW - 1) / GW * GW;
    }
    for (int j = j1; j < nsub; j += GW) {
        float r[8];
        residual8_any<DT, DK, DDT>(c, sm, j, lane, rc, r);
        const float incl = warp_incl_scan(sum8(r));
        if (lane == 31 && walk_check(j < (c.V + kSub - 1) / kSub, sm, DBG_INDEX)) {
            subsum[j] = incl;
            wsum.add(incl);
        }
    }

    if (!total && CL == 1) {
        __syncthreads();
        return;
    }
    if (total && lane == 31) sm.wtot[warp] = wsum.value();
    __syncthreads();
    if (total && warp == 0) {
        double t = lane < kWarps ? sm.wtot[lane] : 0.0;
#pragma unroll
        for (int o = kWarps / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) {
            if (CL == 1)
                sm.total = t;
            else
                sm.ctot = t;
        }
    }
    if (CL == 1) {
        __syncthreads();
        return;
    }
    // Clusters: gather the other CTAs' sub-tile sums and shares of the total.
    cluster_sync();
    for (int j = jlo + (int)threadIdx.x; j < nsub; j += kThreads) {
        const int own = ((j - jlo) % GW) / kWarps;
        if (own != rank) subsum[j] = ld_cluster_f32(cluster_addr(subsum + j, own));
    }
    if (total && threadIdx.x == 0) {
        double t = 0.0;
        for (int r = 0; r < CL; ++r) t += ld_cluster_f64(cluster_addr(&sm.ctot, r));
        sm.total = t;
    }
    cluster_sync();
}

// Largest token with r > 0 in sub-tiles [jlo, jhi) (warp 0), from the stored sub-tile sums:
// the fallback when rounding leaves tau at the very end of the range. -1 if the residual is
// zero there.
template <int DT, int DK, int DDT>
__device__ int last_positive(const Ctx &c, const Smem &sm, const float *subsum, int jlo,
                             int jhi) {
    const int lane = threadIdx.x & 31;
    int jl = -1;
    for (int j = jlo + lane; j < jhi; j += 32)
        if (subsum[j] > 0.f) jl = j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) jl = max(jl, shfl_xor(jl, o));
    if (jl < 0) return -1;
    float r[8];
    int rc = 0;
    residual8_any<DT, DK, DDT>(c, sm, jl, lane, rc, r);
    int lk = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (r[q] > 0.f) lk = jl * kSub + lane * 8 + q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lk = max(lk, shfl_xor(lk, o));
    return lk;
}

// Inverse CDF over the stored sub-tile sums of [jlo, jhi) (warp 0; default: the whole row):
// the bonus token for tau = u * (sum of the range), or for the given tau_abs >= 0 (relative to
// the start of the range); -1 when the residual sums to zero there. One loop narrows the range
// 32 candidates at a time -- groups of consecutive sub-tiles (each lane's group summed with
// compensation), then single sub-tiles -- and a last step searches the 32 lanes x 8 elements
// of the chosen sub-tile. All of it is float arithmetic: every term is a non-negative mass, so
// a prefix formed by a compensated lane sum and a 32-wide scan is within about 7 float
// roundings (4e-7 relative) of its value, inside the 1e-6 * S margin draws are compared on.
// The walk's warp executes this code once per draw, and instruction fetch dominates such cold
// code on this part (the no-instruction stall): one loop body serving every level keeps it
// short. When rounding leaves tau at or past the end of the range, each level takes its last
// candidate with mass, so the draw is the range's last token with r > 0.
template <int DT, int DK, int DDT>
__device__ int bonus_search(const Ctx &c, const Smem &sm, const float *subsum, float u,
                            int jlo = 0, int jhi = -1, double tau_abs = -1.0) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    if (jhi < 0) jhi = (c.V + kSub - 1) / kSub;
    int j0 = jlo, n = jhi - jlo;
    float tau = (float)tau_abs;   // negative: u * (the range's total), set below
    for (bool top = true; top || n > 1; top = false) {
        const int w = (n + 31) / 32;   // sub-tiles per candidate
        const int a = j0 + min(lane * w, n), z = j0 + min(lane * w + w, n);
        KSum g;
        for (int j = a; j < z; ++j) g.add(subsum[j]);
        const float m = g.s - g.c;
        const float incl = warp_incl_scan(m);
        if (top) {
            const float tot = __shfl_sync(full, incl, 31);
            if (!(tot > 0.f)) return -1;
            if (tau < 0.f) tau = u * tot;
        }
        float excl = __shfl_up_sync(full, incl, 1);
        if (lane == 0) excl = 0.f;
        const unsigned hit = __ballot_sync(full, incl > tau);
        int l;
        if (hit) {
            l = __ffs(hit) - 1;
        } else {   // rounding: tau at or past the end; follow the last candidate with mass
            const unsigned pos = __ballot_sync(full, m > 0.f);
            if (!pos) return last_positive<DT, DK, DDT>(c, sm, subsum, jlo, jhi);
            l = 31 - __clz(pos);
            tau = INFINITY;
        }
        tau -= __shfl_sync(full, excl, l);
        j0 = __shfl_sync(full, a, l);
        n = __shfl_sync(full, z, l) - j0;
    }
    const int js = j0;

    // the chosen sub-tile: its 32 lanes x 8 elements (the pass's arithmetic), read again
    const float tr = tau;
    float r[8];
    int rc = 0;
    residual8_any<DT, DK, DDT>(c, sm, js, lane, rc, r);
    const float inc = warp_incl_scan(sum8(r));
    float exf = __shfl_up_sync(full, inc, 1);
    if (lane == 0) exf = 0.f;
    int hitk = -1, lastk = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q) lastk = r[q] > 0.f ? js * kSub + lane * 8 + q : lastk;
    const unsigned b2 = __ballot_sync(full, inc > tr);
    if (b2 != 0) {
        const int l = __ffs(b2) - 1;
        if (lane == l) {
            float part = exf;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                part += r[q];
                if (hitk < 0 && r[q] > 0.f && part > tr) hitk = js * kSub + lane * 8 + q;
            }
            if (hitk < 0) hitk = lastk;
        }
        hitk = __shfl_sync(full, hitk, l);
    }
    if (hitk < 0) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lastk = max(lastk, shfl_xor(lastk, o));
        hitk = lastk >= 0 ? lastk : last_positive<DT, DK, DDT>(c, sm, subsum, jlo, jhi);
    }
    return hitk;
}

// Point drafts: choose the row chunk holding the bonus draw from the chunk partials of the
// stop row (warp 0). The residual mass of chunk q is its sum rescaled to the row max minus
// e_t of the rejected tokens inside it; tau = u * (total). Stores the chunk and tau relative
// to the chunk's start in sm.cpick / sm.ctau. The partials carry float32 rounding of the whole
// row's mass, so when the rejected tokens held half of it or more, that rounding could move
// tau by more than the residual's own precision: then sm.cpick = -1 and the caller sums the
// residual over the whole row instead (as it does when no chunk has mass). (Summing only the
// chunks holding rejected tokens exactly, as the walk's re-sums do, was measured here: no
// faster on deep walks and slower on the common path, whose registers it disturbed.)
__device__ void chunk_pick(const Ctx &c, Smem &sm, const float2 *part, int nc, float u) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    double P = 0.0, M = 0.0;
    if (lane < nc) {
        const float2 pq = part[lane];
        const int lo = row_chunk_sub(lane, c.V, nc) * kSub;
        const int hi = lane == nc - 1 ? c.V : row_chunk_sub(lane + 1, c.V, nc) * kSub;
        P = pq.y > 0.f ? (double)(pq.y * ex2((pq.x + c.negm) * c.k)) : 0.0;
        double mq = P;
        for (int i = 0; i < sm.nR; ++i) {
            const int t = sm.R[i];
            if (t >= lo && t < hi) mq -= (double)sm.RE[i];
        }
        M = mq > 0.0 ? mq : 0.0;
    }
    // float from here on: at most 8 non-negative terms, each within one rounding of its
    // float64 value, so the scan's prefixes are within a few float roundings of S
    const float Mf = (float)M;
    const float incl = warp_incl_scan(Mf);
    const float S = __shfl_sync(full, incl, 31);
    float Ptot = (float)P;   // only compared with S / 2
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ptot += __shfl_xor_sync(full, Ptot, o);
    float excl = __shfl_up_sync(full, incl, 1);
    if (lane == 0) excl = 0.f;
    int pick = -1;
    float tau = 0.f;
    if (S > 0.f && S >= 0.5f * Ptot) {
        tau = u * S;
        const unsigned hit = __ballot_sync(full, lane < nc && incl > tau);
        const unsigned pos = __ballot_sync(full, lane < nc && Mf > 0.f);
        pick = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
        if (pick >= 0) tau = fmaxf(tau - __shfl_sync(full, excl, pick), 0.f);
    }
    if (lane == 0) {
        sm.cpick = pick;
        sm.ctau = tau;
    }
    __syncwarp();
}

// After a heavy rejection the residual mass of the node's row is summed exactly only where it
// has to be: over the chunks holding rejected tokens (marked in sm.cmask), while the other
// chunks' mass comes from their partials (float32 rounding of their own, untouched mass),
// summed into sm.ckeep (warp 0).
__device__ void chunk_marks(const Ctx &c, Smem &sm, const float2 *part, int nc) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    double P = 0.0;
    bool has = false;
    if (lane < nc) {
        const float2 pq = part[lane];
        const int lo = row_chunk_sub(lane, c.V, nc) * kSub;
        const int hi = lane == nc - 1 ? c.V : row_chunk_sub(lane + 1, c.V, nc) * kSub;
        P = pq.y > 0.f ? (double)(pq.y * ex2((pq.x + c.negm) * c.k)) : 0.0;
        for (int i = 0; i < sm.nR; ++i) has |= sm.R[i] >= lo && sm.R[i] < hi;
    }
    const unsigned marks = __ballot_sync(full, has);
    double keep = has ? 0.0 : P;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) keep += __shfl_xor_sync(full, keep, o);
    if (lane == 0) {
        sm.cmask = marks;
        sm.ckeep = keep;
    }
    __syncwarp();
}

// Point drafts: the bonus token for tau (relative to the start of the chunk's sub-tiles
// [jlo, jhi)), drawn without a search by one warp. Warp w streams the contiguous sub-tiles
// [jlo + w per, jlo + (w + 1) per) (per <= draw_subs sub-tiles of a 16-byte aligned row),
// holds their raw vectors in registers, and publishes their totals; in the row's ragged last
// sub-tile (V a multiple of the vector width) the vectors past V are skipped. After one barrier
// every warp forms the same prefix of the 16 block totals; the warp whose block holds tau
// locates the sub-tile among its own totals and the token among its registers (the sub-tile's
// 32 lanes x 8 elements, scanned with the pass's arithmetic). Float sums throughout (see
// bonus_search). When rounding leaves tau at or past the chunk's end, every level follows its
// last candidate with mass: the draw is the chunk's last token with r > 0. Returns the token
// (-1 when the chunk has no mass); all threads call it, and it ends synchronised.
template <int DT>
__device__ int chunk_draw(const Ctx &c, Smem &sm, int jlo, int jhi, float tau) {
    constexpr int K = draw_subs<DT>();
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = jhi - jlo;
    const int per = (n + kWarps - 1) / kWarps;
    const int a = jlo + min(warp * per, n), z = jlo + min(warp * per + per, n);
    // The row's ragged last sub-tile (V a multiple of the vector width here): vectors at or
    // past V are not loaded and their elements get no mass. `ragged` is warp-uniform.
    const bool ragged = z * kSub > c.V;
    uint4 za[K], zb[K];
#pragma unroll
    for (int k = 0; k < K; ++k)
        if (a + k < z) fetch_below<DT>(c.zrow, (a + k) * kSub + lane * 8, ragged ? c.V : INT_MAX,
                                       za[k], zb[k]);
    // Rejected tokens inside this warp's block are rare: test the whole block once, and zero
    // them per sub-tile only then.
    bool anyR = false;
    for (int i = lane; i < sm.nR; i += 32) anyR |= sm.R[i] >= a * kSub && sm.R[i] < z * kSub;
    anyR = __any_sync(full, anyR);
    // The lane sums of all sub-tiles first, then their butterflies level by level, so that the
    // K reductions overlap instead of running one after another (same sums, same order).
    float t[K];
    int rc = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        t[k] = 0.f;
        if (a + k < z) {
            float zs[8], ds[8], r[8];
            shifted8<DT>(za[k], zb[k], c.negm, zs);
            residual8<DRAFT_POINT>(c, sm, zs, ds, r);
            if (anyR) zero_rejected(sm, a + k, lane, rc, r);
            if (ragged) mask_past(r, (a + k) * kSub + lane * 8, c.V);
            t[k] = sum8(r);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < K; ++k) t[k] += __shfl_xor_sync(full, t[k], o);   // same in all lanes
    }
    float wsum = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (a + k < z) {
            if (lane == 0) sm.dsub[warp][k] = t[k];
            wsum += t[k];
        }
    }
    if (lane == 0) sm.dtot[warp] = wsum;
    if (lane == 0 && threadIdx.x == 0) sm.bonus = -1;
    __syncthreads();
    // every warp: the same prefix of the block totals, and the block holding tau
    const float bt = lane < kWarps ? sm.dtot[lane] : 0.f;
    const float incl = warp_incl_scan(bt);
    float excl = __shfl_up_sync(full, incl, 1);
    if (lane == 0) excl = 0.f;
    const unsigned hit = __ballot_sync(full, lane < kWarps && incl > tau);
    const unsigned pos = __ballot_sync(full, lane < kWarps && bt > 0.f);
    int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    float tr = hit ? tau : INFINITY;
    if (warp == owner) {
        tr -= __shfl_sync(full, excl, owner);
        // the sub-tile: first with its running total past tr (else the last with mass)
        int ks = -1, kl = -1;
        float pre = 0.f, prel = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (a + k < z && ks < 0) {
                const float t = sm.dsub[warp][k];
                if (pre + t > tr) {
                    ks = k;
                } else {
                    if (t > 0.f) {
                        kl = k;
                        prel = pre;
                    }
                    pre += t;
                }
            }
        }
        if (ks < 0) {
            ks = kl;
            pre = prel;
            tr = INFINITY;
        }
        int tok = -1;
        if (ks >= 0) {
            uint4 xa = za[0], xb = zb[0];
#pragma unroll
            for (int k = 1; k < K; ++k)
                if (k == ks) {
                    xa = za[k];
                    xb = zb[k];
                }
            const int js = a + ks;
            float zs[8], ds[8], r[8];
            int rc2 = 0;
            shifted8<DT>(xa, xb, c.negm, zs);
            residual8<DRAFT_POINT>(c, sm, zs, ds, r);
            zero_rejected(sm, js, lane, rc2, r);
            if (ragged) mask_past(r, js * kSub + lane * 8, c.V);
            const float trs = tr - pre;
            const float inc = warp_incl_scan(sum8(r));
            float exf = __shfl_up_sync(full, inc, 1);
            if (lane == 0) exf = 0.f;
            int lastk = -1;
#pragma unroll
            for (int q = 0; q < 8; ++q) lastk = r[q] > 0.f ? js * kSub + lane * 8 + q : lastk;
            const unsigned b2 = __ballot_sync(full, inc > trs);
            if (b2 != 0) {
                const int l = __ffs(b2) - 1;
                if (lane == l) {
                    float part = exf;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        part += r[q];
                        if (tok < 0 && r[q] > 0.f && part > trs) tok = js * kSub + lane * 8 + q;
                    }
                    if (tok < 0) tok = lastk;
                }
                tok = __shfl_sync(full, tok, l);
            }
            if (tok < 0) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) lastk = max(lastk, shfl_xor(lastk, o));
                tok = lastk;
            }
        }
        if (lane == 0) sm.bonus = tok;
    }
    __syncthreads();
    return sm.bonus;
}

// ---- the walk (warp 0) ---------------------------------------------------------------------

struct WalkState {
    unsigned long long kids;   // children of the current node not tested yet (bit = node)
    double base, sub;          // point drafts: denominator = base - sub (unnormalised e)
    // Dense drafts: decisions are taken on p and q scaled by S * S_q (S, S_q: the sums of the
    // node's target and draft rows; S_q = 1 for draft probabilities), which needs no
    // division: p S S_q = e_t S_q and q S S_q = e_q S, both exact products in float64. The
    // residual levels are linear in that scale, and u < r / q compares scale-free.
    double mul_p, mul_q;
    int node, L, st, await;
    bool entering, just_summed;
    bool stats_ready;          // lazy walks: the current node's statistics are in shared memory
};

// Point drafts, on entering a node whose children are all among nodes 1..31: every child's
// test at once instead of one child per step (warp 0; lane i holds node i). Children are
// visited in ascending node index; a child repeating an earlier sibling's token is rejected
// outright (that token is already rejected); for the others, the rejected mass before child c
// is the sum of e_t over the distinct tokens of the earlier siblings (a float64 warp scan in
// node order), and c is accepted iff u[c] (S - that mass) < e_t(c), the step-by-step rule. The
// sweep stops at the first child that is accepted or whose denominator fell below S / 16 (the
// exact re-sum then runs first, as in the step-by-step walk). The tokens of the children
// before it enter the rejected list R (ascending, with their e_t) and their mass w.sub.
// Returns the accepted child, or -1 with w.kids holding the children not tested yet.
__device__ int sibling_sweep(WalkState &w, Smem &sm) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const unsigned kids = (unsigned)w.kids;
    const bool k = (kids >> lane) & 1u;
    const int t = k ? sm.tok[lane] : -1 - lane;   // distinct keys for non-children
    // every lane takes part in the match (a warp-wide instruction: none may skip it)
    const unsigned same = __match_any_sync(full, t);
    const bool d = k && (same & ((1u << lane) - 1u)) != 0u;
    const float f = sm.ec[lane];
    const bool live = k && !d;
    const double incl = warp_incl_scan_d(live ? (double)f : 0.0);
    double x = __shfl_up_sync(full, incl, 1);   // rejected mass before this child
    if (lane == 0) x = 0.0;
    const double n = w.base - x;
    const bool h = live && n < w.base * (1.0 / 16.0);
    const bool acc = live && !h && (double)sm.u[lane] * n < (double)f;
    const unsigned stop = __ballot_sync(full, h || acc);
    const int first = stop ? __ffs(stop) - 1 : 32;
    // rejected list: the distinct tokens before `first`, ranked by value
    const bool r = live && lane < first;
    const unsigned rl = __ballot_sync(full, r);
    int rank = 0;
    for (unsigned m = rl; m; m &= m - 1u) rank += __shfl_sync(full, t, __ffs(m) - 1) < t;
    __syncwarp();
    if (r && walk_check(rank < kMaxN, sm, DBG_WALK)) {
        sm.R[rank] = t;
        sm.RE[rank] = f;
    }
    if (lane == 0) sm.nR = __popc(rl);
    __syncwarp();
    w.sub = __shfl_sync(full, first < 32 ? x : incl, first < 32 ? first : 31);
    w.kids = first < 32 ? w.kids & (~0ull << first) : 0ull;
    const unsigned accs = __ballot_sync(full, acc);
    return first < 32 && ((accs >> first) & 1u) ? first : -1;
}

// Advances the walk until it needs a pass over the vocabulary or ends; returns the command.
// Executed by all lanes of warp 0 with identical state.
template <int DK, bool LAZY>
__device__ int advance(WalkState &w, Smem &sm, int N) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    if (w.await == CMD_PASS_SR) {
        w.base = sm.total;
        w.sub = 0.0;
        w.just_summed = true;
    } else if (w.await == CMD_STATS) {
        w.stats_ready = true;
    } else if (w.await == CMD_PASS_Z) {
        const double Z = sm.total;
        if (lane == 0) {
            sm.zinv[sm.nlev] = Z > 0.0 ? 1.0 / Z : 0.0;
            sm.invZ[sm.nlev] = Z > 0.0 ? (float)(1.0 / Z) : 0.f;
            sm.nlev += 1;
            sm.pending = 0;
        }
        __syncwarp();
    }
    w.await = CMD_NONE;
    for (;;) {
        if (w.st) return CMD_DONE;
        if (w.entering) {
            const unsigned b0 =
                __ballot_sync(full, lane >= 1 && lane < N && sm.par[lane] == w.node);
            const unsigned b1 = __ballot_sync(full, lane + 32 < N && sm.par[lane + 32] == w.node);
            w.kids = ((unsigned long long)b1 << 32) | b0;
            if (LAZY && !w.stats_ready) {
                w.await = CMD_STATS;   // stream the node's row(s) first
                return CMD_STATS;
            }
            if (sm.flags[w.node] || (DK != DRAFT_POINT && w.kids && sm.dflags[w.node])) {
                w.st = SPEC_REQ_BAD_ROW;
                continue;
            }
            w.base = (double)sm.s[w.node];
            w.sub = 0.0;
            w.just_summed = false;
            if (DK != DRAFT_POINT && w.kids) {
                w.mul_p = DK == DRAFT_LOGITS ? (double)sm.sq[w.node] : 1.0;
                w.mul_q = (double)sm.s[w.node];
            }
            __syncwarp();
            if (lane == 0) {
                sm.nR = 0;
                sm.nlev = 0;
                sm.pending = 0;
            }
            __syncwarp();
            w.entering = false;
            if constexpr (DK == DRAFT_POINT) {
                if (w.kids && (w.kids >> 32) == 0ull) {
                    const int c = sibling_sweep(w, sm);
                    if (c > 0) {   // accepted: move to it
                        if (!walk_check(w.L < N - 1 && c < N, sm, DBG_WALK)) {
                            w.st = SPEC_REQ_INTERNAL;
                            continue;
                        }
                        if (lane == 0) sm.path[w.L] = c;
                        __syncwarp();
                        w.L += 1;
                        w.node = c;
                        w.entering = true;
                        w.stats_ready = false;
                        continue;
                    }
                }
            }
        }
        if (w.kids == 0) return CMD_BONUS;
        if (DK != DRAFT_POINT && sm.pending) {
            w.await = CMD_PASS_Z;   // normalise the residual the last rejection left
            return CMD_PASS_Z;
        }
        const int c = __ffsll((long long)w.kids) - 1;
        const double uc = (double)sm.u[c];
        bool accept;
        if (DK == DRAFT_POINT) {
            const int t = sm.tok[c];
            const int nR = sm.nR;
            const int r0 = lane < nR ? sm.R[lane] : INT_MAX;
            const int r1 = lane + 32 < nR ? sm.R[lane + 32] : INT_MAX;
            const bool dup = __any_sync(full, r0 == t || r1 == t);
            if (dup) {
                accept = false;
            } else {
                const double denom = w.base - w.sub;
                if (!w.just_summed && denom < w.base * (1.0 / 16.0)) {
                    w.await = CMD_PASS_SR;   // most of the mass is rejected: re-sum exactly
                    return CMD_PASS_SR;
                }
                accept = uc * denom < (double)sm.ec[c];   // u < e_t / denom
            }
            if (!accept) {
                if (!dup && !walk_check(nR < kMaxN, sm, DBG_WALK)) {
                    w.st = SPEC_REQ_INTERNAL;
                    continue;
                }
                if (!dup) {
                    const int pos = __popc(__ballot_sync(full, r0 < t)) +
                                    __popc(__ballot_sync(full, r1 < t));
                    const float e0v = lane < nR ? sm.RE[lane] : 0.f;
                    const float e1v = lane + 32 < nR ? sm.RE[lane + 32] : 0.f;
                    __syncwarp();
                    if (lane < nR && lane >= pos) {
                        sm.R[lane + 1] = r0;
                        sm.RE[lane + 1] = e0v;
                    }
                    if (lane + 32 < nR && lane + 32 >= pos) {
                        sm.R[lane + 33] = r1;
                        sm.RE[lane + 33] = e1v;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        sm.R[pos] = t;
                        sm.RE[pos] = sm.ec[c];
                        sm.nR = nR + 1;
                    }
                    __syncwarp();
                    w.sub += (double)sm.ec[c];
                    w.just_summed = false;
                }
                w.kids &= w.kids - 1;
                continue;
            }
        } else {
            const double p = (double)sm.ec[c] * w.mul_p;   // p S S_q
            const double q = (double)sm.eqc[c] * w.mul_q;  // q S S_q
            double r = p;
            const int nlev = sm.nlev;
            for (int l = 0; l < nlev; ++l)
                if (sm.zinv[l] > 0.0) r = fmax(r - q, 0.0) * sm.zinv[l];
            accept = uc * q < r;
            if (!accept) {
                __syncwarp();
                if (lane == 0) sm.pending = 1;
                __syncwarp();
                w.kids &= w.kids - 1;
                continue;
            }
        }
        if (!walk_check(w.L < N - 1 && c >= 1 && c < N, sm, DBG_WALK)) {
            w.st = SPEC_REQ_INTERNAL;
            continue;
        }
        __syncwarp();
        if (lane == 0) sm.path[w.L] = c;
        __syncwarp();
        w.L += 1;
        w.node = c;
        w.entering = true;
        w.stats_ready = false;
    }
}

// Lazy walks, target row: the row-statistics stream's per-element arithmetic over one row,
// split into kLazyChunks contiguous chunks, one per warp (lanes interleaved). Every
// chunk's (max, sum) goes to sm.cpart, so a bonus drawn from this row sums only one chunk.
// Results land in sm.part_out (m, s, flags). All threads call it; it ends synchronised.
template <int DT>
__device__ void lazy_row_pass(const char *row, int64_t V, float k, Smem &sm, uint4 *ring) {
    using namespace rowpass;
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kEpv = 16 / kEsz;
    constexpr int kGroup = kThreads / kLazyChunks;   // threads per chunk
    constexpr int kWpg = kWarps / kLazyChunks;       // warps per chunk
    static_assert(kWpg >= 1 && kLazyChunks <= 32, "lazy chunks");
    constexpr int kUnroll = SPEC_LAZY_UNROLL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Acc a = acc_init();
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    int64_t head = (int64_t)((16 - (addr & 15)) & 15) / kEsz;
    if (head > V) head = V;
    const int nv = (int)((V - head) / kEpv);
    const int64_t tail0 = head + (int64_t)nv * kEpv;
    const bool aligned = head == 0;
    const int g = tid / kGroup, gt = tid - g * kGroup;
    const int v1 = row_chunk_vec(g + 1, nv, V, aligned, kEpv, kLazyChunks);
    if (g == 0 && gt < head) proc_scalar<ROW_SAMPLE>(a, load_elem<DT>(row, gt), gt, k);
    const uint4 *vb = reinterpret_cast<const uint4 *>(row + head * kEsz);
    int i = row_chunk_vec(g, nv, V, aligned, kEpv, kLazyChunks) + gt;
    constexpr int D = SPEC_LAZY_RING;
    if (D > 0 && ring && aligned) {
        // A ring of this thread's own slots: D copies in flight; each step waits for the
        // oldest (cp.async.wait_group), takes it and refills its slot with the vector D steps
        // ahead. The thread reads back only its own slots, so no barrier is needed, and it
        // visits its vectors in the same order as the register loop below. Slot d of thread t
        // sits at d * kThreads + t, so a warp's 16-byte accesses fall in distinct banks.
        uint4 *slots = ring + threadIdx.x;
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int id = i + d * kGroup;
            if (id < v1 && walk_check(id < nv, sm, DBG_INDEX))
                cp_async16(slots + d * kThreads, vb + id);
            cp_async_commit();
        }
        for (int d = 0; i < v1; i += kGroup, d = d + 1 == D ? 0 : d + 1) {
            cp_async_wait<(D > 0 ? D - 1 : 0)>();
            const uint4 w = slots[d * kThreads];
            const int in = i + D * kGroup;
            if (in < v1 && walk_check(in < nv, sm, DBG_INDEX))
                cp_async16(slots + d * kThreads, vb + in);
            cp_async_commit();
            const int e0 = (int)head + i * kEpv;
            if (DT == 1)
                proc_bf16<ROW_SAMPLE>(a, w, e0, k);
            else
                proc_f32<ROW_SAMPLE>(a, w, e0, k);
        }
        cp_async_wait<0>();
    }
    for (; i + (kUnroll - 1) * kGroup < v1; i += kUnroll * kGroup) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            w[u] = walk_check(i + u * kGroup < nv, sm, DBG_INDEX) ? ldg_stream(vb + i + u * kGroup)
                                                                   : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int e0 = (int)head + (i + u * kGroup) * kEpv;
            if (DT == 1)
                proc_bf16<ROW_SAMPLE>(a, w[u], e0, k);
            else
                proc_f32<ROW_SAMPLE>(a, w[u], e0, k);
        }
    }
    for (; i < v1; i += kGroup) {
        const uint4 w = walk_check(i < nv, sm, DBG_INDEX) ? ldg_stream(vb + i)
                                                           : make_uint4(0, 0, 0, 0);
        const int e0 = (int)head + i * kEpv;
        if (DT == 1)
            proc_bf16<ROW_SAMPLE>(a, w, e0, k);
        else
            proc_f32<ROW_SAMPLE>(a, w, e0, k);
    }
    if (g == kLazyChunks - 1 && tail0 + gt < V) {
        const int idx = (int)(tail0 + gt);
        proc_scalar<ROW_SAMPLE>(a, load_elem<DT>(row, idx), idx, k);
    }
    Part p{a.m, a.s0 + a.s1, a.arg, a.flags};
    p = warp_merge<ROW_SAMPLE>(p, k);
    if (lane == 0) sm.part[warp] = p;
    __syncthreads();
    if (warp == 0) {
        p = lane < kWarps ? sm.part[lane] : Part{-INFINITY, 0.f, kNone, 0};
#pragma unroll
        for (int o = 1; o < kWpg; o <<= 1) p = merge<ROW_SAMPLE>(p, shfl_part(p, o), k);
        if (lane < kWarps && lane % kWpg == 0) sm.cpart[lane / kWpg] = make_float2(p.m, p.s);
#pragma unroll
        for (int o = kWpg; o < 32; o <<= 1) p = merge<ROW_SAMPLE>(p, shfl_part(p, o), k);
        if (p.m == INFINITY) p.flags |= F_POSINF;
        if (p.m == -INFINITY) p.flags |= F_ALLNEG;
        if (lane == 0) sm.part_out = p;
    }
    __syncthreads();
}

// Lazy walks: the statistics of the node's target row (and, for dense drafts of an inner
// node, of its draft row) with the same per-element arithmetic as the row-statistics
// kernel, plus e_t at the children's tokens. All threads call it; it ends synchronised.
template <int DT, int DK, int DDT>
__device__ void lazy_stats(const SampleWalkParams &P, Smem &sm, size_t base, int nd,
                           uint4 *ring) {
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kDDT = DK == DRAFT_LOGITS ? DDT : 0;
    constexpr int kDEsz = kDDT == 1 ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int N = P.N;
    const int64_t V = P.V;
    const float k = P.k;
    const char *zrow = reinterpret_cast<const char *>(P.logits) + (base + nd) * (size_t)V * kEsz;
    int cc[2] = {-1, -1};
    float zc[2] = {0.f, 0.f};
    if (warp == 0) {
        bool any = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = lane + 32 * h;
            if (c >= 1 && c < N && sm.par[c] == nd) {
                any = true;
                cc[h] = c;
                zc[h] = load_elem<DT>(zrow, sm.tok[c]);   // tokens were validated
            }
        }
        const bool kids = __any_sync(0xffffffffu, any);
        if (lane == 0) sm.haskids = kids;
    }
    lazy_row_pass<DT>(zrow, V, k, sm, ring);
    const rowpass::Part p = sm.part_out;
    if (threadIdx.x == 0) sm.cpart_node = nd;
    if (warp == 0) {
        const float negm = p.m == -INFINITY ? 0.f : -p.m;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (cc[h] >= 0) sm.ec[cc[h]] = ex2((zc[h] + negm) * k);
        if (lane == 0) {
            sm.m[nd] = p.m;
            sm.s[nd] = p.s;
            sm.flags[nd] = p.flags;
        }
    }
    if (DK != DRAFT_POINT && sm.haskids) {
        const char *drow =
            reinterpret_cast<const char *>(P.draft) + (base + nd) * (size_t)V * kDEsz;
        float dc[2] = {0.f, 0.f};
        if (warp == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (cc[h] >= 0) dc[h] = load_elem<kDDT>(drow, sm.tok[cc[h]]);
        }
        const rowpass::Part q =
            rowpass::cta_row_stats<kDDT, DK == DRAFT_LOGITS ? ROW_SAMPLE : ROW_PROBS, kThreads,
                                   4>(drow, V, k, sm.part, &sm.part_out);
        if (warp == 0) {
            const float negmq = q.m == -INFINITY ? 0.f : -q.m;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (cc[h] >= 0)
                    sm.eqc[cc[h]] = DK == DRAFT_LOGITS ? ex2((dc[h] + negmq) * k) : dc[h];
            if (lane == 0) {
                sm.mq[nd] = q.m;
                sm.sq[nd] = q.s;
                sm.dflags[nd] = q.flags;
            }
        }
    }
    __syncthreads();
}

template <int DT, int DK, int DDT>
__device__ __forceinline__ Ctx node_ctx(const SampleWalkParams &P, const Smem &sm, size_t base,
                                        int nd) {
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kDEsz = DK == DRAFT_LOGITS ? (DDT == 1 ? 2 : 4) : 4;
    Ctx c;
    c.V = (int)P.V;
    c.k = P.k;
    c.zrow = reinterpret_cast<const char *>(P.logits) + (base + nd) * (size_t)P.V * kEsz;
    c.negm = -sm.m[nd];
    c.invS = 1.f / sm.s[nd];
    c.zvec = (reinterpret_cast<uintptr_t>(c.zrow) & 15) == 0;
    c.drow = DK != DRAFT_POINT
                 ? reinterpret_cast<const char *>(P.draft) + (base + nd) * (size_t)P.V * kDEsz
                 : nullptr;
    c.dvec = DK != DRAFT_POINT && (reinterpret_cast<uintptr_t>(c.drow) & 15) == 0;
    c.negmq = DK == DRAFT_LOGITS ? -sm.mq[nd] : 0.f;
    c.invSq = DK == DRAFT_LOGITS ? 1.f / sm.sq[nd] : 1.f;
    c.useq = DK != DRAFT_POINT && (sm.nlev > 0 || sm.pending);
    return c;
}

// Point drafts: the chunk partials of the current node's target row, when the walk has them
// (eager: from the row-statistics kernel; lazy: from the pass over that row) and the row is
// 16-byte aligned; else null.
template <bool LAZY>
__device__ __forceinline__ const float2 *node_part(const SampleWalkParams &P, const Smem &sm,
                                                   const Ctx &c) {
    if (!c.zvec) return nullptr;
    if (LAZY) return sm.cpart_node == sm.node ? sm.cpart : nullptr;
    return P.chunk ? sm.epart[sm.node] : nullptr;
}

// Point drafts fit 64 registers (2 CTAs per SM); dense drafts keep more live values.
// LAZY: no row-statistics kernel ran; the walk streams only the rows it visits.
// CL: CTAs per request (eager walks), launched as one thread-block cluster per request; they
// share every vocabulary pass, and the leading CTA writes the outputs.
template <int DT, int DK, int DDT, bool LAZY, int CL = 1>
__global__ void __launch_bounds__(kThreads, DK == DRAFT_POINT ? 2 : 1)
    walk_sample_kernel(SampleWalkParams P) {
    static_assert(CL == 1 || CL == 2 || CL == 4 || CL == 8, "cluster size");
    static_assert(!LAZY || CL == 1, "lazy walks run one CTA per request");
    __shared__ Smem sm;
    extern __shared__ float subsum[];   // sub-tile sums of the current pass
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = CL == 1 ? (int)blockIdx.x : (int)blockIdx.x / CL;
    const int N = P.N;
    const size_t base = (size_t)b * N;
    const int nb = node_budget(P.n_active, b, N);   // nodes >= nb do not exist in this call

    if (tid < N && tid >= nb) {   // never a child of any node
        sm.par[tid] = -2;
        sm.tok[tid] = -1;
    }
    if (tid < nb) {
        sm.par[tid] = P.parent[base + tid];
        sm.tok[tid] = P.tok[base + tid];
    }
    if (tid <= N) sm.u[tid] = P.uniforms[(size_t)b * (N + 1) + tid];
    // Eager walks are launched to overlap the row-statistics kernel's end: its results are
    // read only after it has completed (the tree and uniforms above come from before it).
    if (!LAZY) grid_dep_wait();
    if (!LAZY && DK == DRAFT_POINT && P.chunk && tid < nb * kRowChunks)
        (&sm.epart[0][0])[tid] = P.chunk[base * kRowChunks + tid];
    if (tid < nb && !LAZY) {
        sm.flags[tid] = P.flags[base + tid];
        sm.s[tid] = P.s[base + tid];
        sm.m[tid] = P.m[base + tid];
        sm.ec[tid] = tid >= 1 ? P.pc[base + tid] : 0.f;
        if (DK != DRAFT_POINT) {
            sm.dflags[tid] = P.dflags[base + tid];
            sm.eqc[tid] = tid >= 1 ? P.qc[base + tid] : 0.f;
            if (DK == DRAFT_LOGITS) {
                sm.sq[tid] = P.sq[base + tid];
                sm.mq[tid] = P.mq[base + tid];
            }
        }
    }
    if (tid == 0) {
        sm.nR = 0;
        sm.nlev = 0;
        sm.pending = 0;
        sm.bonus = -1;
        sm.cpart_node = -1;
        sm.dbgv = 0;
    }
    __syncthreads();

    WalkState w;
    w.kids = 0;
    w.base = w.sub = 0.0;
    w.mul_p = w.mul_q = 1.0;
    w.node = 0;
    w.L = 0;
    w.st = 0;
    w.await = CMD_NONE;
    w.entering = true;
    w.just_summed = false;
    w.stats_ready = false;
    if (warp == 0) {
        // Request checks in the oracle's order: parents, draft tokens, uniforms.
        bool bp = false, bt = false, bu = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            if (i < nb) {
                const int p = sm.par[i];
                bp |= i == 0 ? p != -1 : (p < 0 || p >= i);
                if (i >= 1) bt |= sm.tok[i] < 0 || sm.tok[i] >= P.V;
            }
            // uniform slots of the existing children, and the bonus slot N
            const int iu = i + 1;
            if (iu < nb || iu == N) bu |= !(sm.u[iu] >= 0.f && sm.u[iu] < 1.f);
        }
        w.st = nb == 0                ? SPEC_REQ_BAD_BUDGET
               : __any_sync(full, bp) ? SPEC_REQ_BAD_PARENT
               : __any_sync(full, bt) ? SPEC_REQ_BAD_TOKEN
               : __any_sync(full, bu) ? SPEC_REQ_BAD_UNIFORM
                                      : 0;
    }

    int cmd = CMD_NONE;
    for (;;) {
        if (warp == 0) {
            cmd = advance<DK, LAZY>(w, sm, N);
            if (lane == 0) {
                sm.cmd = cmd;
                sm.node = w.node;
                sm.L = w.L;
                sm.st = w.st;
            }
        }
        __syncthreads();
        cmd = lead<CL>(sm, sm.cmd);
        if (cmd == CMD_DONE || cmd == CMD_BONUS) break;
        if (LAZY && cmd == CMD_STATS) {
            // rows in host memory are read with plain loads: cp.async copies from host memory
            // ran at half the rate over the host link (0.90 against 0.41 ms per large-tree call)
            lazy_stats<DT, DK, DDT>(
                P, sm, base, sm.node,
                P.host_rows ? nullptr : reinterpret_cast<uint4 *>(subsum + lazy_ring_offset(P.V)));
            continue;
        }
        const Ctx c = node_ctx<DT, DK, DDT>(P, sm, base, sm.node);
        // Eager point drafts (a heavy rejection): re-sum only the chunks holding rejected
        // tokens, one pass per chunk, the other chunks from their partials. One call site for
        // every pass keeps the walk's registers from spilling. (Lazy walks re-sum the whole
        // row: the extra state spilled in their pass loop and slowed every lazy call.)
        constexpr int nc = LAZY ? kLazyChunks : kRowChunks;
        unsigned mk = 0;
        if constexpr (DK == DRAFT_POINT && !LAZY) {
            const float2 *part = node_part<LAZY>(P, sm, c);
            if (part) {
                if (warp == 0) chunk_marks(c, sm, part, nc);
                __syncthreads();
                mk = sm.cmask;
                if (__popc(mk) > 2) mk = 0;   // more chunk passes than one row pass would cost
            }
        }
        const bool chunked = mk != 0;
        double acc = chunked ? sm.ckeep : 0.0;
        do {
            int jlo = 0, jhi = INT_MAX;
            if (chunked) {
                const int q = __ffs(mk) - 1;
                mk &= mk - 1;
                jlo = row_chunk_sub(q, c.V, nc);
                jhi = row_chunk_sub(q + 1, c.V, nc);
            }
            residual_pass<DT, DK, DDT, CL>(c, sm, subsum, jlo, jhi);
            acc += sm.total;
        } while (mk);
        if (chunked) {
            __syncthreads();   // every thread has read the last pass's total
            if (tid == 0) sm.total = acc;
            __syncthreads();
        }
    }

    if (cmd == CMD_BONUS) {
        const float ub = sm.u[N];
        bool drawn = false;
        if constexpr (DK == DRAFT_POINT) {
            // One chunk instead of the row: locate the chunk from the chunk partials of the
            // stop row (the row-statistics kernel's, or those of the lazy pass over it), then
            // sum and search only its sub-tiles. Rows that are not 16-byte aligned have no
            // partials.
            static_assert(CL == 1, "point drafts run one CTA per request");
            const Ctx c = node_ctx<DT, DK, DDT>(P, sm, base, sm.node);
            constexpr int nc = LAZY ? kLazyChunks : kRowChunks;
            const float2 *part = node_part<LAZY>(P, sm, c);
            int q = -1;
            if (part) {
                if (warp == 0) chunk_pick(c, sm, part, nc, ub);
                __syncthreads();
                q = sm.cpick;
                if (!walk_check(q < nc, sm, DBG_INDEX)) q = -1;
            }
            if (q >= 0) {
                const int jlo = row_chunk_sub(q, c.V, nc), jhi = row_chunk_sub(q + 1, c.V, nc);
                if (jhi - jlo <= kWarps * draw_subs<DT>() &&
                    (jhi <= c.V / kSub || c.V % (DT == 1 ? 8 : 4) == 0)) {
                    // sub-tiles that the warps can hold (an eighth of the row for eager walks,
                    // a sixteenth for lazy ones; the last may be ragged): drawn without a
                    // search
                    drawn = chunk_draw<DT>(c, sm, jlo, jhi, (float)sm.ctau) >= 0;
                } else {
                    residual_pass<DT, DK, DDT>(c, sm, subsum, jlo, jhi, false);
                    if (warp == 0) {
                        const int v = bonus_search<DT, DK, DDT>(c, sm, subsum, ub, jlo, jhi,
                                                                sm.ctau);
                        if (lane == 0) sm.bonus = v;
                    }
                    __syncthreads();
                    drawn = sm.bonus >= 0;
                }
            }
        }
        for (int attempt = 0; attempt < 3 && !drawn; ++attempt) {
            const Ctx c = node_ctx<DT, DK, DDT>(P, sm, base, sm.node);
            residual_pass<DT, DK, DDT, CL>(c, sm, subsum);
            if (warp == 0) {
                const int v = bonus_search<DT, DK, DDT>(c, sm, subsum, ub);
                if (lane == 0) sm.bonus = v;
            }
            __syncthreads();
            if (lead<CL>(sm, sm.bonus) >= 0) break;
            // The residual sums to zero. Dense: the last level is degenerate (target and draft
            // agree to rounding): keep the previous level. Point: every token with mass was
            // rejected through rounding: draw from the node's target row.
            __syncthreads();
            if (tid == 0) {
                if (sm.pending) {
                    sm.pending = 0;
                } else {
                    sm.nR = 0;
                    sm.nlev = 0;
                }
            }
            __syncthreads();
        }
    }
    __syncthreads();
    if constexpr (kDebug) {
        // The accepted path is a chain of parent links from the root; the bonus is a token
        // and, for point drafts, not one of the stop node's rejected tokens; no row statistics
        // of this request failed a check. Any violation turns the result into
        // SPEC_REQ_INTERNAL.
        if (tid == 0) {
            int v = sm.dbgv;
            if (sm.st == 0) {
                int prev = 0;
                for (int j = 0; j < sm.L; ++j) {
                    const int nd = sm.path[j];
                    if (nd < 1 || nd >= N || sm.par[nd] != prev) v |= DBG_WALK;
                    prev = nd >= 0 && nd < N ? nd : 0;
                }
                if (!(sm.bonus >= 0 && sm.bonus < P.V)) v |= DBG_WALK;
                if (DK == DRAFT_POINT)
                    for (int i = 0; i < sm.nR; ++i)
                        if (sm.R[i] == sm.bonus) v |= DBG_WALK;
            }
            if (sm.st == SPEC_REQ_INTERNAL) v |= DBG_WALK;
            if (P.dbg) {
                if (v) atomicOr(P.dbg + b, v);
                if (P.dbg[b]) v |= P.dbg[b];
            }
            if (v) sm.st = SPEC_REQ_INTERNAL;
        }
        __syncthreads();
    }
    if (CL > 1 && cluster_rank() != 0) return;   // the leading CTA writes the outputs

    // Compaction.
    const int fst = sm.st;
    const int fL = sm.L;
    const int fb = sm.bonus;
    for (int j = tid; j < N; j += kThreads) {
        int ot = -1, kv = -1;
        if (fst == 0) {
            if (j < fL)
                ot = sm.tok[sm.path[j]];
            else if (j == fL)
                ot = fb;
            if (j == 0)
                kv = 0;
            else if (j <= fL)
                kv = sm.path[j - 1];
        }
        P.out.out_tokens[base + j] = ot;
        P.out.kv_commit[base + j] = kv;
    }
    if (tid == 0) {
        P.out.accept_len[b] = fst ? 0 : fL;
        P.out.bonus[b] = fst ? -1 : fb;
        P.out.status[b] = fst;
    }
}

template <int DT, int DK, int DDT>
cudaError_t launch_ws(const SampleWalkParams &p, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)subsum_floats(p.V);   // sub-tile sums
    if (!p.lazy) {
        const dim3 block(kThreads);
        // Point drafts pass over one chunk of the stop row at most: a cluster's barriers would
        // cost more than splitting that pass saves, so they keep one CTA per request.
        if constexpr (DK != DRAFT_POINT) {
            if (p.cluster > 1) {
                cudaError_t e;
                if (p.cluster == 8)
                    e = launch_dependent_cluster(walk_sample_kernel<DT, DK, DDT, false, 8>,
                                                 dim3(p.B * 8), block, smem, st, 8, p);
                else if (p.cluster == 4)
                    e = launch_dependent_cluster(walk_sample_kernel<DT, DK, DDT, false, 4>,
                                                 dim3(p.B * 4), block, smem, st, 4, p);
                else
                    e = launch_dependent_cluster(walk_sample_kernel<DT, DK, DDT, false, 2>,
                                                 dim3(p.B * 2), block, smem, st, 2, p);
                // A device or partition that cannot co-schedule the cluster refuses its launch
                // configuration (nothing was launched): clear that error and run one CTA per
                // request instead. Other errors are returned.
                if (e != cudaErrorNotSupported && e != cudaErrorInvalidClusterSize &&
                    e != cudaErrorLaunchOutOfResources)
                    return e;
                cudaGetLastError();
            }
        }
        return launch_dependent(walk_sample_kernel<DT, DK, DDT, false>, dim3(p.B), block, smem,
                                st, p);
    }
    // lazy walks: the sub-tile sums, then the ring of the row passes
    const size_t lsmem = sizeof(float) * (size_t)lazy_ring_offset(p.V) + kLazyRingBytes;
    const cudaError_t e = cudaFuncSetAttribute(walk_sample_kernel<DT, DK, DDT, true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)lsmem);
    if (e != cudaSuccess) return e;
    walk_sample_kernel<DT, DK, DDT, true><<<p.B, kThreads, lsmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace
}  // namespace specv
