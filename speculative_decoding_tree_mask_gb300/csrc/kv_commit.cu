// KV commit: copy the K/V of the root and the accepted nodes into a paged KV cache.
//
// IluvatarLabs/vllm PR #3 ("commit_draft_kernel"): masked draft K/V are copied into the paged
// cache (NHD or HND layout; fp16/bf16/fp32 sources; a cache of the source type or fp8 with a
// scale; masked entries return early). EmbodiInfer PR #11 (commits 938fe7b and 41dcd00) keeps
// per-row KV buffers and commits only the new tokens. Slot j of request b (kv_commit[b][j],
// j = 0..accept_len[b]: the root, then the accepted nodes in path order) goes to sequence
// position seq_pos[b] + j:
//   block = block_table[b][p / block_size], offset = p % block_size,
//   NHD cache [num_blocks, block_size, H, D], HND cache [num_blocks, H, block_size, D].
// fp8 caches hold cvt.rn.satfinite(x / scale) (x / scale rounded to float32 first); the scale
// is one value per tensor or one per source token (b, node).
// One CTA per (slot, request); CTAs of slots beyond accept_len return at once. Each thread
// moves 8 elements per step (one or two 16-byte loads, one 16- or 8-byte store).

#include <cuda_fp16.h>

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kThreads = 128;

template <int SRC>
__device__ __forceinline__ float src_elem(const void *p, size_t i) {
    if (SRC == 0) return __ldg(reinterpret_cast<const float *>(p) + i);
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
    if (SRC == 1) return __uint_as_float(uint32_t(h) << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t fp8x2(float a, float b, int kind) {
    uint16_t r;
    if (kind == 1)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
    return r;
}

// One scalar element src[si] -> cache[di].
template <int SRC, int CACHE>
__device__ __forceinline__ void put1(const void *src, size_t si, void *dst, size_t di,
                                     float scale) {
    if (CACHE == 0) {
        if (SRC == 0)
            reinterpret_cast<float *>(dst)[di] = __ldg(reinterpret_cast<const float *>(src) + si);
        else
            reinterpret_cast<unsigned short *>(dst)[di] =
                __ldg(reinterpret_cast<const unsigned short *>(src) + si);
    } else {
        const float q = __fdiv_rn(src_elem<SRC>(src, si), scale);
        reinterpret_cast<uint8_t *>(dst)[di] = (uint8_t)(fp8x2(q, 0.f, CACHE) & 0xff);
    }
}

// Eight elements src[si..si+8) -> cache[di..di+8) (16-byte aligned source and destination).
template <int SRC, int CACHE>
__device__ __forceinline__ void put8(const void *src, size_t si, void *dst, size_t di,
                                     float scale) {
    constexpr int kSrcBytes = SRC == 0 ? 4 : 2;
    const char *sp = reinterpret_cast<const char *>(src) + si * kSrcBytes;
    if (CACHE == 0) {
        if (SRC == 0) {
            const uint4 a = ldg_stream(reinterpret_cast<const uint4 *>(sp));
            const uint4 b = ldg_stream(reinterpret_cast<const uint4 *>(sp) + 1);
            uint4 *dp = reinterpret_cast<uint4 *>(reinterpret_cast<char *>(dst) + di * 4);
            dp[0] = a;
            dp[1] = b;
        } else {
            const uint4 a = ldg_stream(reinterpret_cast<const uint4 *>(sp));
            *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(dst) + di * 2) = a;
        }
        return;
    }
    float x[8];
    if (SRC == 0) {
        const uint4 a = ldg_stream(reinterpret_cast<const uint4 *>(sp));
        const uint4 b = ldg_stream(reinterpret_cast<const uint4 *>(sp) + 1);
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
        x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    } else {
        const uint4 a = ldg_stream(reinterpret_cast<const uint4 *>(sp));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (SRC == 1) {
                x[2 * q] = bf_lo(w[q]);
                x[2 * q + 1] = bf_hi(w[q]);
            } else {
                const __half2 hv = *reinterpret_cast<const __half2 *>(&w[q]);
                const float2 f = __half22float2(hv);
                x[2 * q] = f.x;
                x[2 * q + 1] = f.y;
            }
        }
    }
    uint2 o;
    uint16_t c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        c[q] = fp8x2(__fdiv_rn(x[2 * q], scale), __fdiv_rn(x[2 * q + 1], scale), CACHE);
    o.x = uint32_t(c[0]) | (uint32_t(c[1]) << 16);
    o.y = uint32_t(c[2]) | (uint32_t(c[3]) << 16);
    *reinterpret_cast<uint2 *>(reinterpret_cast<char *>(dst) + di) = o;
}

template <int SRC, int CACHE, bool VEC>
__global__ void __launch_bounds__(kThreads) kv_commit_kernel(KvCommitParams P) {
    const int j = blockIdx.x, b = blockIdx.y;
    const int N = P.N;
    const int32_t *kv = P.kv_commit + (size_t)b * N;
    const int L = P.accept_len[b];
    const int root = kv[0];
    // Slot 0's CTA decides the request's status (all slots checked there, no write races).
    if (j == 0 && threadIdx.x == 0 && P.status) {
        int st = 0;
        if (root >= 0) {
            for (int jj = 0; jj <= L && jj < N; ++jj) {
                const int p = P.seq_pos[b] + jj;
                const int bi = p >= 0 ? p / P.block_size : -1;
                const int blk = (bi >= 0 && bi < P.max_blocks) ? P.block_table[(size_t)b * P.max_blocks + bi] : -1;
                const int node = kv[jj];
                if (blk < 0 || blk >= P.num_blocks || node < 0 || node >= N) st = SPEC_REQ_BAD_SLOT;
            }
        }
        P.status[b] = st;
    }
    if (root < 0 || j > L) return;   // failed verification or slot not accepted
    const int node = kv[j];
    if (node < 0 || node >= N) return;
    const int p = P.seq_pos[b] + j;
    if (p < 0) return;
    const int bi = p / P.block_size;
    if (bi >= P.max_blocks) return;
    const int blk = P.block_table[(size_t)b * P.max_blocks + bi];
    if (blk < 0 || blk >= P.num_blocks) return;
    const int off = p - bi * P.block_size;
    const int H = P.H, D = P.D, HD = H * D;
    const size_t si = P.scale_per_token ? (size_t)b * N + node : 0;
    const float ks = P.k_scale ? P.k_scale[si] : 1.f;
    const float vs = P.v_scale ? P.v_scale[si] : 1.f;
    const size_t sbase = ((size_t)b * N + node) * (size_t)HD;
    const int step = VEC ? 8 : 1;
    for (int e = threadIdx.x * step; e < HD; e += kThreads * step) {
        const int h = e / D, d = e - h * D;
        const size_t di = P.layout == 0
                              ? (((size_t)blk * P.block_size + off) * H + h) * (size_t)D + d
                              : (((size_t)blk * H + h) * P.block_size + off) * (size_t)D + d;
        if (VEC) {
            put8<SRC, CACHE>(P.src_k, sbase + e, P.cache_k, di, ks);
            put8<SRC, CACHE>(P.src_v, sbase + e, P.cache_v, di, vs);
        } else {
            put1<SRC, CACHE>(P.src_k, sbase + e, P.cache_k, di, ks);
            put1<SRC, CACHE>(P.src_v, sbase + e, P.cache_v, di, vs);
        }
    }
}

template <int SRC, int CACHE>
cudaError_t launch_kc(const KvCommitParams &p, bool vec, cudaStream_t st) {
    const dim3 grid(p.N, p.B);
    if (vec)
        kv_commit_kernel<SRC, CACHE, true><<<grid, kThreads, 0, st>>>(p);
    else
        kv_commit_kernel<SRC, CACHE, false><<<grid, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <int SRC>
cudaError_t launch_src(const KvCommitParams &p, bool vec, cudaStream_t st) {
    if (p.cache_kind == 1) return launch_kc<SRC, 1>(p, vec, st);
    if (p.cache_kind == 2) return launch_kc<SRC, 2>(p, vec, st);
    return launch_kc<SRC, 0>(p, vec, st);
}

}  // namespace

cudaError_t launch_kv_commit(const KvCommitParams &p, bool vec, cudaStream_t st) {
    if (p.B <= 0) return cudaSuccess;
    if (p.src_dtype == 1) return launch_src<1>(p, vec, st);
    if (p.src_dtype == 2) return launch_src<2>(p, vec, st);
    return launch_src<0>(p, vec, st);
}

}  // namespace specv
