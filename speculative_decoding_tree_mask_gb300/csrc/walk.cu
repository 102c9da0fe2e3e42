// Tree walk, bonus draw and accepted-path compaction.
//
// EmbodiInfer PR #11 "perf(activevln): grammar-trie speculation and lossless throughput",
// commit 4b728e2: greedy decoding keeps the argmax path; sampling uses standard rejection
// sampling against the draft (SpecInfer-style on a trie), so the output distribution is the
// target's. Both walks start at the root and visit children in ascending node index.
//
// Greedy: one warp per request; the per-row argmax and flags of the request (N <= 64) sit in
// registers, children are found with one ballot per level.
//
// Sampling: one CTA per request. Thread 0 runs the walk on scalars gathered by the row-stats
// kernel (e_t = 2^((z_t - m) log2(e)/T) at every child token, the row sums S, and for dense
// drafts the same for the draft rows). Whenever a decision needs a sum over the vocabulary the
// whole CTA streams the row once ("pass"):
//   * point drafts: p(t) / sum_{v not in R} p(v) is formed as e_t / (S - sum_{R} e); when the
//     rejected mass exceeds 15/16 of the denominator the remainder is re-summed exactly;
//   * dense drafts: after a rejection with siblings left, Z = sum_v max(r(v) - q(v), 0)
//     normalises the next residual level;
//   * bonus: the residual at the stop node is summed per 256-element sub-tile (warp scans,
//     sub-tile sums kept in shared memory), the sub-tile holding tau = u * S is located, and
//     that sub-tile is re-read to find the token.
// Sub-tile sums, the located sub-tile's in-warp scan and the final element search use the same
// float32 arithmetic in the same order, so the search always ends on a token with r(v) > 0.

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

// ------------------------------------------------------------------------------------------
// greedy walk
// ------------------------------------------------------------------------------------------

constexpr int kGreedyWarps = 4;

__global__ void __launch_bounds__(32 * kGreedyWarps) walk_greedy_kernel(GreedyWalkParams P) {
    const unsigned full = 0xffffffffu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kGreedyWarps + warp;
    if (b >= P.B) return;
    const int N = P.N;
    const size_t base = (size_t)b * N;

    int par[2], tk[2], ag[2], fl[2];
    bool bad_par = false, bad_tok = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < N) {
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
    int st = __any_sync(full, bad_par) ? 1 : (__any_sync(full, bad_tok) ? 2 : 0);

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

// ------------------------------------------------------------------------------------------
// sampling walk
// ------------------------------------------------------------------------------------------

constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kSub = 256;           // elements per sub-tile: 32 lanes x 8
constexpr int kPassUnroll = 4;      // sub-tiles in flight per warp

enum { CMD_NONE = 0, CMD_DONE, CMD_BONUS, CMD_PASS_SR, CMD_PASS_Z };

struct WalkSmem {
    int par[kMaxN], tok[kMaxN], flags[kMaxN], dflags[kMaxN];
    float ec[kMaxN];     // e_t of each child in its parent's target row
    float eqc[kMaxN];    // draft: e_q at each child token (probabilities: q itself)
    float s[kMaxN], m[kMaxN], sq[kMaxN], mq[kMaxN];
    float u[kMaxN + 1];
    int path[kMaxN];
    int R[kMaxN];        // rejected tokens at the current node, ascending
    float invZ[kMaxN];   // dense: 1 / Z of each normalised residual level (0: level kept)
    double zval[kMaxN];  // dense: Z of each level (thread 0's decisions)
    int nR, nlev, pending;
    int cmd, node, L, st, bonus, jstar, last_pos;
    double total, tau_rem;
    double wtot[kWalkWarps];
    int wlast[kWalkWarps];
};

struct RowCtx {
    const char *zrow;    // target row of the node
    const char *drow;    // draft row of the node (dense)
    float negm, invS, negmq, invSq, k;
    int V;
    bool zvec, dvec;     // rows 16-byte aligned
    bool useq;           // dense residual levels present: the draft row is read
};

// 8 consecutive elements starting at e0 (e0 % 8 == 0); beyond V they read as 0 / -inf.
template <int DT>
__device__ __forceinline__ void load8(const char *row, int e0, int V, bool vec, float (&x)[8],
                                      float fill) {
    if (vec && e0 + 8 <= V) {
        if (DT == 1) {
            const uint4 w = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 8);
            x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
            x[4] = bf_lo(w.z); x[5] = bf_hi(w.z); x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
        } else {
            const uint4 w0 = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4);
            const uint4 w1 = ldg_stream(reinterpret_cast<const uint4 *>(row) + e0 / 4 + 1);
            x[0] = __uint_as_float(w0.x); x[1] = __uint_as_float(w0.y);
            x[2] = __uint_as_float(w0.z); x[3] = __uint_as_float(w0.w);
            x[4] = __uint_as_float(w1.x); x[5] = __uint_as_float(w1.y);
            x[6] = __uint_as_float(w1.z); x[7] = __uint_as_float(w1.w);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = e0 + q < V ? load_elem<DT>(row, e0 + q) : fill;
    }
}

// Residual values r(v) of the 8 elements at e0 for the current pass.
template <int DT, int DK, int DDT>
__device__ __forceinline__ void residual8(const RowCtx &c, const WalkSmem &sm, int e0,
                                          const float (&z)[8], const float (&d)[8],
                                          int &rcur, float (&r)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float e = ex2((z[q] + c.negm) * c.k);
        if (DK == DRAFT_POINT) {
            r[q] = e;
        } else {
            float x = e * c.invS;
            if (c.useq) {
                const float qv =
                    DK == DRAFT_LOGITS ? ex2((d[q] + c.negmq) * c.k) * c.invSq : d[q];
                for (int l = 0; l < sm.nlev; ++l)
                    if (sm.invZ[l] > 0.f) x = fmaxf(x - qv, 0.f) * sm.invZ[l];
                if (sm.pending) x = fmaxf(x - qv, 0.f);
            }
            r[q] = x;
        }
        if (e0 + q >= c.V) r[q] = 0.f;
    }
    if (DK == DRAFT_POINT) {
        // zero the rejected tokens (sorted): skip those below this lane's range
        while (rcur < sm.nR && sm.R[rcur] < e0) ++rcur;
        for (int i = rcur; i < sm.nR && sm.R[i] < e0 + 8; ++i) r[sm.R[i] - e0] = 0.f;
    }
}

// One pass over the node's residual: every warp sums its sub-tiles (optionally storing the
// sub-tile sums), the CTA total lands in sm.total and the largest index with r > 0 in
// sm.last_pos. Called by all threads; ends synchronised.
template <int DT, int DK, int DDT>
__device__ void residual_pass(const RowCtx &c, WalkSmem &sm, float *subsum, bool store) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsub = (c.V + kSub - 1) / kSub;
    double wsum = 0.0;
    int last = -1;
    int rcur = 0;
    for (int j0 = warp; j0 < nsub; j0 += kWalkWarps * kPassUnroll) {
        float z[kPassUnroll][8], d[kPassUnroll][8];
#pragma unroll
        for (int uu = 0; uu < kPassUnroll; ++uu) {
            const int j = j0 + uu * kWalkWarps;
            if (j < nsub) {
                const int e0 = j * kSub + lane * 8;
                load8<DT>(c.zrow, e0, c.V, c.zvec, z[uu], -INFINITY);
                if (DK == DRAFT_LOGITS && c.useq)
                    load8<DDT>(c.drow, e0, c.V, c.dvec, d[uu], -INFINITY);
                if (DK == DRAFT_PROBS_F32 && c.useq)
                    load8<0>(c.drow, e0, c.V, c.dvec, d[uu], 0.f);
            }
        }
#pragma unroll
        for (int uu = 0; uu < kPassUnroll; ++uu) {
            const int j = j0 + uu * kWalkWarps;
            if (j >= nsub) break;
            const int e0 = j * kSub + lane * 8;
            float r[8];
            residual8<DT, DK, DDT>(c, sm, e0, z[uu], d[uu], rcur, r);
            float ls = r[0];
#pragma unroll
            for (int q = 1; q < 8; ++q) ls += r[q];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (r[q] > 0.f) last = e0 + q;
            const float incl = warp_incl_scan(ls);
            if (lane == 31) {
                if (store) subsum[j] = incl;
                wsum += (double)incl;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last = max(last, shfl_xor(last, o));
    if (lane == 31) {
        sm.wtot[warp] = wsum;
        sm.wlast[warp] = last;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        int lp = -1;
        for (int w = 0; w < kWalkWarps; ++w) {
            t += sm.wtot[w];
            lp = max(lp, sm.wlast[w]);
        }
        sm.total = t;
        sm.last_pos = lp;
    }
    __syncthreads();
}

// Inverse CDF over the stored sub-tile sums (warp 0): the bonus token for uniform u, or -1
// when the residual sums to zero.
template <int DT, int DK, int DDT>
__device__ int bonus_search(const RowCtx &c, WalkSmem &sm, const float *subsum, float u) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int nsub = (c.V + kSub - 1) / kSub;
    const int cs = (nsub + 31) / 32;
    const int lo = min(lane * cs, nsub), hi = min(lo + cs, nsub);
    double lt = 0.0;
    for (int j = lo; j < hi; ++j) lt += (double)subsum[j];
    const double incl = warp_incl_scan_d(lt);
    const double S = __shfl_sync(full, incl, 31);
    if (!(S > 0.0)) return -1;
    double excl = __shfl_up_sync(full, incl, 1);
    if (lane == 0) excl = 0.0;
    const double tau = (double)u * S;
    const unsigned ball = __ballot_sync(full, incl > tau);
    int js = -1;
    double pref = 0.0;
    if (ball != 0) {
        const int owner = __ffs(ball) - 1;
        if (lane == owner) {
            pref = excl;
            int lastpos_j = -1;
            double lastP = 0.0, run = excl;
            for (int j = lo; j < hi; ++j) {
                if (subsum[j] > 0.f) {
                    lastpos_j = j;
                    lastP = run;
                }
                if (run + (double)subsum[j] > tau) {
                    js = j;
                    pref = run;
                    break;
                }
                run += (double)subsum[j];
            }
            if (js < 0) {
                js = lastpos_j;
                pref = lastP;
            }
        }
        js = __shfl_sync(full, js, owner);
        pref = __shfl_sync(full, pref, owner);
    }
    if (js < 0) return sm.last_pos;   // rounding left tau at the very end of the row

    // Re-read sub-tile js and find the element (same arithmetic as the pass).
    const double tr = tau - pref;
    const int e0 = js * kSub + lane * 8;
    float z[8], d[8];
    load8<DT>(c.zrow, e0, c.V, c.zvec, z, -INFINITY);
    if (DK == DRAFT_LOGITS && c.useq) load8<DDT>(c.drow, e0, c.V, c.dvec, d, -INFINITY);
    if (DK == DRAFT_PROBS_F32 && c.useq) load8<0>(c.drow, e0, c.V, c.dvec, d, 0.f);
    float r[8];
    int rcur = 0;
    residual8<DT, DK, DDT>(c, sm, e0, z, d, rcur, r);
    float ls = r[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) ls += r[q];
    const float inc = warp_incl_scan(ls);
    float exf = __shfl_up_sync(full, inc, 1);
    if (lane == 0) exf = 0.f;
    int lastk = -1;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (r[q] > 0.f) lastk = e0 + q;
    int hit = -1;
    const unsigned b2 = __ballot_sync(full, (double)inc > tr);
    if (b2 != 0) {
        const int owner = __ffs(b2) - 1;
        if (lane == owner) {
            float part = 0.f;
            for (int q = 0; q < 8; ++q) {
                part = q == 0 ? r[0] : part + r[q];
                if ((double)exf + (double)part > tr) {
                    hit = e0 + q;
                    break;
                }
            }
            if (hit < 0) hit = lastk;
        }
        hit = __shfl_sync(full, hit, owner);
    }
    if (hit < 0) {
        int lk = lastk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lk = max(lk, shfl_xor(lk, o));
        hit = lk >= 0 ? lk : sm.last_pos;
    }
    return hit;
}

template <int DT, int DK, int DDT>
__global__ void __launch_bounds__(kWalkThreads) walk_sample_kernel(SampleWalkParams P) {
    __shared__ WalkSmem sm;
    extern __shared__ float subsum[];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const int N = P.N;
    const int V = (int)P.V;
    const size_t base = (size_t)b * N;
    constexpr bool kDense = DK != DRAFT_POINT;
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kDEsz = DK == DRAFT_LOGITS ? (DDT == 1 ? 2 : 4) : 4;

    if (tid < N) {
        sm.par[tid] = P.parent[base + tid];
        sm.tok[tid] = P.tok[base + tid];
        sm.flags[tid] = P.flags[base + tid];
        sm.s[tid] = P.s[base + tid];
        sm.m[tid] = P.m[base + tid];
        sm.ec[tid] = tid >= 1 ? P.pc[base + tid] : 0.f;
        if (kDense) {
            sm.dflags[tid] = P.dflags[base + tid];
            sm.eqc[tid] = tid >= 1 ? P.qc[base + tid] : 0.f;
            if (DK == DRAFT_LOGITS) {
                sm.sq[tid] = P.sq[base + tid];
                sm.mq[tid] = P.mq[base + tid];
            }
        }
    }
    if (tid <= N) sm.u[tid] = P.uniforms[(size_t)b * (N + 1) + tid];
    if (tid == 0) {
        sm.nR = 0;
        sm.nlev = 0;
        sm.pending = 0;
    }
    __syncthreads();

    // Thread 0's walk state (meaningful in thread 0 only).
    int node = 0, L = 0, st = 0, cursor = 1, await = CMD_NONE;
    bool entering = true;
    double dbase = 0.0, dsub = 0.0;
    if (tid == 0) {
        for (int i = 0; i < N && st == 0; ++i) {
            const int p = sm.par[i];
            if (i == 0 ? p != -1 : (p < 0 || p >= i)) st = 1;
        }
        for (int i = 1; i < N && st == 0; ++i)
            if (sm.tok[i] < 0 || sm.tok[i] >= V) st = 2;
        for (int i = 1; i <= N && st == 0; ++i)
            if (!(sm.u[i] >= 0.f && sm.u[i] < 1.f)) st = 4;
    }

    int cmd;
    for (;;) {
        if (tid == 0) {
            cmd = CMD_NONE;
            if (await == CMD_PASS_SR) {
                dbase = sm.total;
                dsub = 0.0;
            } else if (await == CMD_PASS_Z) {
                const double Z = sm.total;
                sm.zval[sm.nlev] = Z;
                sm.invZ[sm.nlev] = Z > 0.0 ? (float)(1.0 / Z) : 0.f;
                sm.nlev += 1;
                sm.pending = 0;
            }
            const bool resumed = await == CMD_PASS_SR;
            await = CMD_NONE;
            bool just_summed = resumed;
            while (cmd == CMD_NONE) {
                if (st) {
                    cmd = CMD_DONE;
                    break;
                }
                if (entering) {
                    bool kids = false;
                    for (int c = node + 1; c < N; ++c) kids |= sm.par[c] == node;
                    if (sm.flags[node] || (kDense && kids && sm.dflags[node])) {
                        st = 3;
                        continue;
                    }
                    dbase = (double)sm.s[node];
                    dsub = 0.0;
                    sm.nR = 0;
                    sm.nlev = 0;
                    sm.pending = 0;
                    cursor = node + 1;
                    entering = false;
                    just_summed = false;
                }
                int c = cursor;
                while (c < N && sm.par[c] != node) ++c;
                if (c >= N) {
                    cmd = CMD_BONUS;
                    break;
                }
                if (kDense && sm.pending) {
                    cmd = CMD_PASS_Z;   // normalise the residual left by the last rejection
                    await = CMD_PASS_Z;
                    break;
                }
                const double uc = (double)sm.u[c];
                bool accept;
                if (!kDense) {
                    const int t = sm.tok[c];
                    bool dup = false;
                    for (int i = 0; i < sm.nR; ++i) dup |= sm.R[i] == t;
                    if (dup) {
                        accept = false;
                    } else {
                        const double denom = dbase - dsub;
                        if (!just_summed && denom < dbase * (1.0 / 16.0)) {
                            cmd = CMD_PASS_SR;   // too much mass rejected: re-sum exactly
                            await = CMD_PASS_SR;
                            break;
                        }
                        accept = uc < (double)sm.ec[c] / denom;
                    }
                    if (!accept) {
                        if (!dup) {
                            int i = sm.nR;
                            while (i > 0 && sm.R[i - 1] > t) {
                                sm.R[i] = sm.R[i - 1];
                                --i;
                            }
                            sm.R[i] = t;
                            sm.nR += 1;
                            dsub += (double)sm.ec[c];
                            just_summed = false;
                        }
                        cursor = c + 1;
                        continue;
                    }
                } else {
                    const double p = (double)sm.ec[c] / (double)sm.s[node];
                    const double q = DK == DRAFT_LOGITS ? (double)sm.eqc[c] / (double)sm.sq[node]
                                                        : (double)sm.eqc[c];
                    double r = p;
                    for (int l = 0; l < sm.nlev; ++l)
                        if (sm.zval[l] > 0.0) r = fmax(r - q, 0.0) / sm.zval[l];
                    accept = uc * q < r;
                    if (!accept) {
                        sm.pending = 1;
                        cursor = c + 1;
                        continue;
                    }
                }
                sm.path[L++] = c;
                node = c;
                entering = true;
            }
            sm.cmd = cmd;
            sm.node = node;
            sm.L = L;
            sm.st = st;
        }
        __syncthreads();
        cmd = sm.cmd;
        if (cmd == CMD_DONE || cmd == CMD_BONUS) break;

        const int nd = sm.node;
        RowCtx c;
        c.V = V;
        c.k = P.k;
        c.zrow = reinterpret_cast<const char *>(P.logits) + (base + nd) * (size_t)V * kEsz;
        c.negm = -sm.m[nd];
        c.invS = 1.f / sm.s[nd];
        c.zvec = (reinterpret_cast<uintptr_t>(c.zrow) & 15) == 0;
        c.drow = kDense ? reinterpret_cast<const char *>(P.draft) + (base + nd) * (size_t)V * kDEsz
                        : nullptr;
        c.dvec = kDense && (reinterpret_cast<uintptr_t>(c.drow) & 15) == 0;
        c.negmq = DK == DRAFT_LOGITS ? -sm.mq[nd] : 0.f;
        c.invSq = DK == DRAFT_LOGITS ? 1.f / sm.sq[nd] : 1.f;
        c.useq = kDense && (sm.nlev > 0 || sm.pending);
        residual_pass<DT, DK, DDT>(c, sm, subsum, false);
    }

    if (cmd == CMD_BONUS) {
        const int nd = sm.node;
        RowCtx c;
        c.V = V;
        c.k = P.k;
        c.zrow = reinterpret_cast<const char *>(P.logits) + (base + nd) * (size_t)V * kEsz;
        c.negm = -sm.m[nd];
        c.invS = 1.f / sm.s[nd];
        c.zvec = (reinterpret_cast<uintptr_t>(c.zrow) & 15) == 0;
        c.drow = kDense ? reinterpret_cast<const char *>(P.draft) + (base + nd) * (size_t)V * kDEsz
                        : nullptr;
        c.dvec = kDense && (reinterpret_cast<uintptr_t>(c.drow) & 15) == 0;
        c.negmq = DK == DRAFT_LOGITS ? -sm.mq[nd] : 0.f;
        c.invSq = DK == DRAFT_LOGITS ? 1.f / sm.sq[nd] : 1.f;
        const float ub = sm.u[N];
        for (int attempt = 0; attempt < 3; ++attempt) {
            c.useq = kDense && (sm.nlev > 0 || sm.pending);
            residual_pass<DT, DK, DDT>(c, sm, subsum, true);
            if (tid < 32) {
                const int v = bonus_search<DT, DK, DDT>(c, sm, subsum, ub);
                if (tid == 0) sm.bonus = v;
            }
            __syncthreads();
            if (sm.bonus >= 0) break;
            // The residual sums to zero. Dense: the last level is degenerate (target and draft
            // agree to rounding), keep the previous level. Point: every token with mass was
            // rejected through rounding; draw from the node's target row.
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

    // Compaction.
    const int fst = sm.st;
    const int fL = sm.L;
    const int fb = sm.bonus;
    for (int j = tid; j < N; j += kWalkThreads) {
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
    const size_t smem = walk_sample_smem(p.V);
    walk_sample_kernel<DT, DK, DDT><<<p.B, kWalkThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t walk_sample_smem(int64_t V) { return sizeof(float) * (size_t)((V + kSub - 1) / kSub); }

cudaError_t launch_walk_greedy(const GreedyWalkParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    const int grid = (p.B + kGreedyWarps - 1) / kGreedyWarps;
    walk_greedy_kernel<<<grid, 32 * kGreedyWarps, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_walk_sample(const SampleWalkParams &p, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    if (p.draft_kind == DRAFT_POINT) {
        if (p.dtype == 1) return launch_ws<1, DRAFT_POINT, 0>(p, st);
        return launch_ws<0, DRAFT_POINT, 0>(p, st);
    }
    if (p.draft_kind == DRAFT_PROBS_F32) {
        if (p.dtype == 1) return launch_ws<1, DRAFT_PROBS_F32, 0>(p, st);
        return launch_ws<0, DRAFT_PROBS_F32, 0>(p, st);
    }
    if (p.dtype == 1) {
        if (p.draft_dtype == 1) return launch_ws<1, DRAFT_LOGITS, 1>(p, st);
        return launch_ws<1, DRAFT_LOGITS, 0>(p, st);
    }
    if (p.draft_dtype == 1) return launch_ws<0, DRAFT_LOGITS, 1>(p, st);
    return launch_ws<0, DRAFT_LOGITS, 0>(p, st);
}

}  // namespace specv
