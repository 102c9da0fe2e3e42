// Per-element row-statistics arithmetic shared by the streaming kernels: the running max,
// lowest-index argmax and temperature-scaled sum of exponentials over one row, merged across
// threads. Used by the one-CTA-per-row stream (row_stats.cu) and by the passes of the lazy
// walks, so both compute every element the same way. Internal to the CUDA path.
#pragma once

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace rowpass {

enum { F_NAN = 1, F_POSINF = 2, F_ALLNEG = 4 };

struct Acc {
    float m;      // running max (never NaN)
    float negm;   // -m once m is finite, else 0
    float s0, s1; // partial sums of 2^((x - m) k)
    int arg;      // lowest index attaining m (kNone before any non -inf element)
    int flags;
};

__device__ __forceinline__ Acc acc_init() {
    Acc a;
    a.m = -INFINITY;
    a.negm = 0.f;
    a.s0 = a.s1 = 0.f;
    a.arg = kNone;
    a.flags = 0;
    return a;
}

// Packed FP32 pairs (two lanes per instruction, each rounded like its scalar form).
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) {
    unsigned long long x, y, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
    unsigned long long x, y, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}

// (2^((x_lo + c) k), 2^((x_hi + c) k)) for the two bf16 of w: widening and the subtraction in
// one mixed-precision add each, the scaling by k as one packed multiply.
__device__ __forceinline__ float2 ex2_bf16_pair(uint32_t w, float c, float k) {
    float d0, d1;
    bf_add2(w, c, d0, d1);
    const float2 t = mul_f32x2(make_float2(d0, d1), make_float2(k, k));
    return make_float2(ex2(t.x), ex2(t.y));
}

template <int MODE>
__device__ __forceinline__ void raise_max(Acc &a, float v, float k) {
    if (MODE == ROW_SAMPLE) {
        if (a.m == -INFINITY) {
            a.s0 = 0.f;
            a.s1 = 0.f;
        } else {
            const float f = ex2((a.m - v) * k);
            a.s0 *= f;
            a.s1 *= f;
        }
    }
    a.m = v;
    a.negm = -v;
}

// One scalar element (head / tail of a misaligned row).
template <int MODE>
__device__ __forceinline__ void proc_scalar(Acc &a, float x, int idx, float k) {
    if (MODE == ROW_PROBS) {
        if (!(x >= 0.f && x < INFINITY)) a.flags |= F_NAN;
        return;
    }
    if (x != x) {
        a.flags |= F_NAN;
    } else if (x > a.m) {
        raise_max<MODE>(a, x, k);
        a.arg = idx;
    }
    if (MODE == ROW_SAMPLE) a.s0 += ex2((x + a.negm) * k);
}

// Eight bf16 values (one 16-byte vector) starting at element e0.
template <int MODE>
__device__ __forceinline__ void proc_bf16(Acc &a, const uint4 w, int e0, float k) {
    const uint32_t mm = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
    const float vmax = fmax_nan(bf_lo(mm), bf_hi(mm));
    if (!(vmax <= a.m)) {
        if (vmax != vmax) {
            a.flags |= F_NAN;
        } else {
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            int j = 7;
#pragma unroll
            for (int q = 3; q >= 0; --q) {
                if (bf_hi(ws[q]) == vmax) j = 2 * q + 1;
                if (bf_lo(ws[q]) == vmax) j = 2 * q;
            }
            raise_max<MODE>(a, vmax, k);
            a.arg = e0 + j;
        }
    }
    if (MODE == ROW_SAMPLE) {
        // Even elements accumulate in s0, odd ones in s1, each as ((e0 + e2) + (e4 + e6)):
        // the multiplies by k and the sums run as packed pairs (half the instructions of the
        // scalar form, with the same roundings in the same order).
        const float2 p0 = ex2_bf16_pair(w.x, a.negm, k), p1 = ex2_bf16_pair(w.y, a.negm, k);
        const float2 p2 = ex2_bf16_pair(w.z, a.negm, k), p3 = ex2_bf16_pair(w.w, a.negm, k);
        const float2 q = add_f32x2(add_f32x2(p0, p1), add_f32x2(p2, p3));
        const float2 s = add_f32x2(make_float2(a.s0, a.s1), q);
        a.s0 = s.x;
        a.s1 = s.y;
    }
}

// Four f32 values (one 16-byte vector) starting at element e0.
template <int MODE>
__device__ __forceinline__ void proc_f32(Acc &a, const uint4 w, int e0, float k) {
    const float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                        __uint_as_float(w.w)};
    if (MODE == ROW_PROBS) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (!(x[q] >= 0.f && x[q] < INFINITY)) a.flags |= F_NAN;
        return;
    }
    const float vmax = fmax_nan(fmax_nan(x[0], x[1]), fmax_nan(x[2], x[3]));
    if (!(vmax <= a.m)) {
        if (vmax != vmax) {
            a.flags |= F_NAN;
        } else {
            int j = 3;
#pragma unroll
            for (int q = 2; q >= 0; --q)
                if (x[q] == vmax) j = q;
            raise_max<MODE>(a, vmax, k);
            a.arg = e0 + j;
        }
    }
    if (MODE == ROW_SAMPLE) {
        // s0 += e0 + e2, s1 += e1 + e3, in packed pairs
        const float2 c = make_float2(a.negm, a.negm), kk = make_float2(k, k);
        const float2 t01 = mul_f32x2(add_f32x2(make_float2(x[0], x[1]), c), kk);
        const float2 t23 = mul_f32x2(add_f32x2(make_float2(x[2], x[3]), c), kk);
        const float2 q = add_f32x2(make_float2(ex2(t01.x), ex2(t01.y)),
                                   make_float2(ex2(t23.x), ex2(t23.y)));
        const float2 s = add_f32x2(make_float2(a.s0, a.s1), q);
        a.s0 = s.x;
        a.s1 = s.y;
    }
}

struct Part {
    float m, s;
    int arg, flags;
};

// Vector idx of a row of n 16-byte vectors. Debug builds check the index first and, when it
// is outside the row, record the violation and return zeros instead of loading.
__device__ __forceinline__ uint4 ldg_checked(const uint4 *row, int idx, int n, int32_t *dbg,
                                             int b) {
    if (!dbg_check(idx >= 0 && idx < n, dbg, b, DBG_INDEX)) return make_uint4(0, 0, 0, 0);
    return ldg_stream(row + idx);
}

// The same, recording a violation in a shared-memory word of the CTA (when given).
__device__ __forceinline__ uint4 ldg_flagged(const uint4 *row, int idx, int n, int *flag) {
    if constexpr (kDebug) {
        if (!(idx >= 0 && idx < n)) {
            if (flag) atomicOr(flag, DBG_INDEX);
            return make_uint4(0, 0, 0, 0);
        }
    }
    return ldg_stream(row + idx);
}

template <int MODE>
__device__ __forceinline__ Part merge(Part x, Part y, float k) {
    Part r;
    r.m = fmaxf(x.m, y.m);
    r.flags = x.flags | y.flags;
    r.arg = x.m > y.m ? x.arg : (y.m > x.m ? y.arg : min(x.arg, y.arg));
    r.s = 0.f;
    if (MODE == ROW_SAMPLE && r.m != -INFINITY)
        r.s = x.s * ex2((x.m - r.m) * k) + y.s * ex2((y.m - r.m) * k);
    return r;
}

// The partial of lane (lane ^ o).
__device__ __forceinline__ Part shfl_part(const Part &p, int o) {
    Part q;
    q.m = shfl_xor(p.m, o);
    q.s = shfl_xor(p.s, o);
    q.arg = shfl_xor(p.arg, o);
    q.flags = shfl_xor(p.flags, o);
    return q;
}

template <int MODE>
__device__ __forceinline__ Part warp_merge(Part p, float k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) p = merge<MODE>(p, shfl_part(p, o), k);
    return p;
}


// One CTA streams one row: returns the merged statistics to every thread. THREADS must match
// blockDim.x; sh_part needs THREADS / 32 entries. Same per-element arithmetic as the
// one-CTA-per-row kernel. Debug builds check every vector index and set DBG_INDEX in the
// shared word *flag (when given) instead of loading outside the row.
template <int DT, int MODE, int THREADS, int UNROLL>
__device__ __forceinline__ Part cta_row_stats(const char *rowp, int64_t V, float k,
                                              Part *sh_part, Part *sh_out,
                                              int *flag = nullptr) {
    constexpr int kEsz = DT == 1 ? 2 : 4;
    constexpr int kEpv = 16 / kEsz;
    constexpr int kW = THREADS / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Acc a = acc_init();
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
    int64_t head = (int64_t)((16 - (addr & 15)) & 15) / kEsz;
    if (head > V) head = V;
    const int64_t nvec = (V - head) / kEpv;
    const int64_t tail0 = head + nvec * kEpv;
    if (tid < head) proc_scalar<MODE>(a, load_elem<DT>(rowp, tid), tid, k);
    const uint4 *vb = reinterpret_cast<const uint4 *>(rowp + head * kEsz);
    const int nv = (int)nvec;
    int i = tid;
    for (; i + (UNROLL - 1) * THREADS < nv; i += UNROLL * THREADS) {
        uint4 w[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) w[u] = ldg_flagged(vb, i + u * THREADS, nv, flag);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int e0 = (int)head + (i + u * THREADS) * kEpv;
            if (DT == 1)
                proc_bf16<MODE>(a, w[u], e0, k);
            else
                proc_f32<MODE>(a, w[u], e0, k);
        }
    }
    for (; i < nv; i += THREADS) {
        const uint4 w = ldg_flagged(vb, i, nv, flag);
        const int e0 = (int)head + i * kEpv;
        if (DT == 1)
            proc_bf16<MODE>(a, w, e0, k);
        else
            proc_f32<MODE>(a, w, e0, k);
    }
    if (tail0 + tid < V) {
        const int idx = (int)(tail0 + tid);
        proc_scalar<MODE>(a, load_elem<DT>(rowp, idx), idx, k);
    }
    Part p{a.m, a.s0 + a.s1, a.arg, a.flags};
    p = warp_merge<MODE>(p, k);
    if (lane == 0) sh_part[warp] = p;
    __syncthreads();
    if (warp == 0) {
        p = lane < kW ? sh_part[lane] : Part{-INFINITY, 0.f, kNone, 0};
        p = warp_merge<MODE>(p, k);
        if (MODE != ROW_PROBS) {
            if (p.m == INFINITY) p.flags |= F_POSINF;
            if (p.m == -INFINITY) p.flags |= F_ALLNEG;
        }
        if (p.arg == kNone) p.arg = 0;
        if (lane == 0) *sh_out = p;
    }
    __syncthreads();
    return *sh_out;
}

}  // namespace rowpass
}  // namespace specv
