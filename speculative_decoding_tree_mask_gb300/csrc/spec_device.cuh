// Device-side helpers of the verification kernels (sm_103a). Internal to the CUDA path.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "spec_internal.h"

namespace specv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kNone = 0x7fffffff;   // "no index yet" in argmax reductions

// Debug flavour (compiled with SPEC_DEBUG): the kernels check the indices they compute and
// the split rows' arrival counters. A failed check sets a bit in the request's debug word
// (a per-request int32 array of the handle) and the offending access is skipped; the walk
// that finishes the request then reports SPEC_REQ_INTERNAL instead of its result. Nothing
// traps. In release builds every check is the constant true and compiles to nothing.
#ifdef SPEC_DEBUG
constexpr bool kDebug = true;
#else
constexpr bool kDebug = false;
#endif
enum { DBG_INDEX = 1, DBG_ARRIVAL = 2, DBG_WALK = 4 };

__device__ __forceinline__ bool dbg_check(bool ok, int32_t *words, int b, int bit) {
    if constexpr (kDebug) {
        if (!ok && words) atomicOr(words + b, bit);
        return ok;
    } else {
        return true;
    }
}

// Number of nodes request b verifies under a node budget: all N without one, the budget when
// it lies in [1, N], and 0 (the request is refused) otherwise.
__device__ __forceinline__ int node_budget(const int32_t *n_active, int b, int N) {
    if (!n_active) return N;
    const int n = n_active[b];
    return n >= 1 && n <= N ? n : 0;
}

// 2^x on the special-function unit (flushes denormal results to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Lane-wise max of two bf16 pairs; a NaN in either operand propagates.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// bf16 halves of a packed word widened to float (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// (x + c) for both bf16 halves of w, widened and added in one rounding each.
__device__ __forceinline__ void bf_add2(uint32_t w, float c, float &d0, float &d1) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %3;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(w), "f"(c));
}

// 16-byte streaming load: read-only path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch. A kernel launched with launch_dependent (spec_internal.h)
// may start while the kernel before it in the stream still runs; grid_dep_wait() returns once
// that kernel has completed and its writes are visible (at once for an ordinary launch).
// grid_dep_launch() lets the next such kernel start launching.
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters (kernels launched with launch_dependent_cluster). cluster_sync() is
// the hardware cluster barrier, taken by every thread of every CTA of the cluster (the
// non-aligned form: warps need not be converged when they reach it). It orders shared-memory
// writes before it with distributed shared-memory reads after it. One CTA may read another's
// shared memory only between two cluster barriers, so that the owner has started and does
// not exit or overwrite the data before the reader is done.
__device__ __forceinline__ int cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\t"
                 "barrier.cluster.wait.acquire;" ::: "memory");
}
// The address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, int rank) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ double ld_cluster_f64(uint32_t a) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t a) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

// Scalar element load as float (bf16 or f32 storage).
template <int DT>
__device__ __forceinline__ float load_elem(const void *row, int64_t i);
template <>
__device__ __forceinline__ float load_elem<0>(const void *row, int64_t i) {
    return __ldg(reinterpret_cast<const float *>(row) + i);
}
template <>
__device__ __forceinline__ float load_elem<1>(const void *row, int64_t i) {
    uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(row) + i);
    return __uint_as_float(uint32_t(h) << 16);
}

template <typename T>
__device__ __forceinline__ T shfl_xor(T v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }

// Inclusive warp scan (fixed association: Hillis-Steele over the 32 lanes).
__device__ __forceinline__ float warp_incl_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__device__ __forceinline__ double warp_incl_scan_d(double x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

}  // namespace specv
