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
// Work is split into units of (slot j, request b, piece of the slot's H*D elements), ordered
// slot-major, so that the slots every request commits (j <= accept_len) come first. A grid of
// 8 CTAs per SM strides over the units: each CTA first reads every request's accepted length
// and position into shared memory (all loads issued before any is used) and stops at the
// deepest accepted slot of the batch, so no CTA works on a slot nobody commits. Per unit the
// node and the cache block are loaded together, the next unit's while this unit's data is in
// flight, and each thread loads all of its K and V elements of the unit (four 16-byte vectors
// of each for 16-bit sources) before it stores any of them. The statuses are checked by the
// CTAs that get the fewest units.

#include <cuda_fp16.h>

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kThreads = 128;
constexpr int kCtasPerSm = 6;   // resident CTAs per SM the register budget allows

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

// Raw source elements of one 8-element vector: one 16-byte load (bf16 / f16) or two (f32).
template <int SRC>
struct Raw8 {
    uint4 a, b;
};

template <int SRC>
__device__ __forceinline__ Raw8<SRC> load8(const void *src, size_t si) {
    constexpr int kSrcBytes = SRC == 0 ? 4 : 2;
    const uint4 *sp =
        reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(src) + si * kSrcBytes);
    Raw8<SRC> r;
    r.a = ldg_stream(sp);
    if (SRC == 0) r.b = ldg_stream(sp + 1);
    return r;
}

// Store one loaded vector at cache element di (16-byte aligned source and destination).
template <int SRC, int CACHE>
__device__ __forceinline__ void store8(const Raw8<SRC> &r, void *dst, size_t di, float scale) {
    if (CACHE == 0) {
        if (SRC == 0) {
            uint4 *dp = reinterpret_cast<uint4 *>(reinterpret_cast<char *>(dst) + di * 4);
            dp[0] = r.a;
            dp[1] = r.b;
        } else {
            *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(dst) + di * 2) = r.a;
        }
        return;
    }
    float x[8];
    if (SRC == 0) {
        x[0] = __uint_as_float(r.a.x); x[1] = __uint_as_float(r.a.y);
        x[2] = __uint_as_float(r.a.z); x[3] = __uint_as_float(r.a.w);
        x[4] = __uint_as_float(r.b.x); x[5] = __uint_as_float(r.b.y);
        x[6] = __uint_as_float(r.b.z); x[7] = __uint_as_float(r.b.w);
    } else {
        const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
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

// 8-element vectors of K (and as many of V) per thread per unit: 128 bytes of loads in
// flight per thread for 16-bit sources, 256 for f32.
template <int SRC>
constexpr int vecs() { return SRC == 0 ? 2 : 4; }
constexpr int kUnitElems = kThreads * 8 * 4;      // elements of K (and of V) per unit
constexpr int kSmemRequests = 4096;               // requests whose (L, position) fit in smem

// Cache element of (slot position `off` in block `blk`, element e of the H*D slot).
__device__ __forceinline__ size_t cache_index(const KvCommitParams &P, int blk, int off, int e) {
    const int h = e / P.D, d = e - h * P.D;
    return P.layout == 0 ? (((size_t)blk * P.block_size + off) * P.H + h) * (size_t)P.D + d
                         : (((size_t)blk * P.H + h) * P.block_size + off) * (size_t)P.D + d;
}

// Debug builds: a source or cache index outside its array is skipped and the request's
// commit status becomes SPEC_REQ_INTERNAL (statuses are combined with atomicMax there, the
// library having zeroed them before the launch). Release builds check nothing.
__device__ __forceinline__ bool kv_index_ok(const KvCommitParams &P, int b, size_t si, size_t di,
                                            int n) {
    if constexpr (kDebug) {
        const size_t HD = (size_t)P.H * P.D;
        const bool ok = si + n <= (size_t)P.B * P.N * HD &&
                        di + n <= (size_t)P.num_blocks * P.block_size * HD;
        if (!ok && P.status) atomicMax(P.status + b, (int)SPEC_REQ_INTERNAL);
        return ok;
    } else {
        return true;
    }
}

// The last slot request b commits: min(accept_len, N - 1), or -1 when its verification
// failed (kv_commit[b][0] < 0) and nothing is written.
__device__ __forceinline__ int last_slot(const KvCommitParams &P, int b) {
    if (P.kv_commit[(size_t)b * P.N] < 0) return -1;
    return min(max(P.accept_len[b], 0), P.N - 1);
}

// One unit of work: slot j of request b, piece `piece` of the slot's H*D elements.
struct Unit {
    int j, b, piece, L, pos;
};

// The request's status: SPEC_REQ_BAD_SLOT if any committed slot maps outside the block table
// or the cache, else 0. One warp, one lane per slot.
__device__ __forceinline__ void request_status(const KvCommitParams &P, int b, int L, int pos,
                                               int lane) {
    bool bad = false;
    for (int jj = lane; jj <= L; jj += 32) {
        const int p = pos + jj;
        const int bi = p >= 0 ? p / P.block_size : -1;
        const int blk =
            (bi >= 0 && bi < P.max_blocks) ? P.block_table[(size_t)b * P.max_blocks + bi] : -1;
        const int node = P.kv_commit[(size_t)b * P.N + jj];
        bad |= blk < 0 || blk >= P.num_blocks || node < 0 || node >= P.N;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        if (kDebug)
            atomicMax(P.status + b, bad ? (int)SPEC_REQ_BAD_SLOT : 0);
        else
            P.status[b] = bad ? SPEC_REQ_BAD_SLOT : 0;
    }
}

template <int SRC, int CACHE, bool VEC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    kv_commit_kernel(KvCommitParams P, int pieces) {
    extern __shared__ int s_req[];   // [2][B]: last slot, position of slot 0 (B <= 4096)
    __shared__ int s_max;
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, N = P.N, G = (int)gridDim.x;
    const bool cached = B <= kSmemRequests;
    int lmax = N - 1;
    if (cached) {
        // Every load of the prologue is issued before any is used: one round trip.
        int m = -1;
        for (int b0 = 0; b0 < B; b0 += 4 * kThreads) {
            int root[4], al[4], ps[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int b = b0 + q * kThreads + tid;
                root[q] = b < B ? __ldg(P.kv_commit + (size_t)b * N) : -1;
                al[q] = b < B ? __ldg(P.accept_len + b) : 0;
                ps[q] = b < B ? __ldg(P.seq_pos + b) : 0;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int b = b0 + q * kThreads + tid;
                if (b < B) {
                    const int l = root[q] < 0 ? -1 : min(max(al[q], 0), N - 1);
                    s_req[b] = l;
                    s_req[B + b] = ps[q];
                    m = max(m, l);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(full, m, o));
        if (tid == 0) s_max = -1;
        __syncthreads();
        if (lane == 0) atomicMax(&s_max, m);
        __syncthreads();
        lmax = s_max;
    }
    // Statuses: request b is checked by warp 0 of CTA G-1-(b mod G), the CTAs that get the
    // fewest copy units; the other warps start copying meanwhile.
    if (P.status && warp == 0)
        for (int b = G - 1 - (int)blockIdx.x; b < B; b += G)
            request_status(P, b, cached ? s_req[b] : last_slot(P, b),
                           cached ? s_req[B + b] : P.seq_pos[b], lane);

    const int HD = P.H * P.D;
    const int64_t per_slot = (int64_t)B * pieces;
    const int64_t units = (int64_t)(max(lmax, 0) + 1) * per_slot;
    // The CTA's next unit at or after u (stride G) that copies something; units when none.
    auto next_live = [&](int64_t u, Unit &x) -> int64_t {
        for (; u < units; u += G) {
            x.j = (int)(u / per_slot);
            const int64_t r = u - (int64_t)x.j * per_slot;
            x.b = (int)(r / pieces);
            x.piece = (int)(r - (int64_t)x.b * pieces);
            x.L = cached ? s_req[x.b] : last_slot(P, x.b);
            if (x.j > x.L) continue;   // failed verification, or a slot it does not commit
            x.pos = cached ? s_req[B + x.b] : P.seq_pos[x.b];
            return u;
        }
        return units;
    };
    // Node and cache block of a unit, loaded together (-1: nothing to copy).
    auto unit_index = [&](const Unit &x, int &node, int &blk) {
        const int p = x.pos + x.j;
        const int bi = p >= 0 ? p / P.block_size : -1;
        node = __ldg(P.kv_commit + (size_t)x.b * N + x.j);
        blk = (bi >= 0 && bi < P.max_blocks)
                  ? __ldg(P.block_table + (size_t)x.b * P.max_blocks + bi)
                  : -1;
    };

    Unit cur;
    int64_t u = next_live(blockIdx.x, cur);
    int node = -1, blk = -1;
    if (u < units) unit_index(cur, node, blk);
    while (u < units) {
        const int p = cur.pos + cur.j;
        const bool live = node >= 0 && node < N && blk >= 0 && blk < P.num_blocks && p >= 0;
        const int off = live ? p - (p / P.block_size) * P.block_size : 0;
        const int b = cur.b;
        const size_t si = P.scale_per_token ? (size_t)b * N + (live ? node : 0) : 0;
        const size_t sbase = ((size_t)b * N + (live ? node : 0)) * (size_t)HD;
        const int e0 = cur.piece * kUnitElems, e1 = min(HD, e0 + kUnitElems);
        const int cblk = blk;
        // The next unit's indices are fetched while this unit's data is in flight.
        Unit nxt;
        const int64_t un = next_live(u + G, nxt);
        if (VEC) {
            // f32 sources: the unit's 4096 elements in two passes of two vectors each
            constexpr int kV = vecs<SRC>();
#pragma unroll
            for (int half = 0; half < 4 / kV; ++half) {
                Raw8<SRC> k[kV], v[kV];
#pragma unroll
                for (int q = 0; q < kV; ++q) {
                    const int e = e0 + (tid + (half * kV + q) * kThreads) * 8;
                    if (live && e < e1 &&
                        kv_index_ok(P, b, sbase + e, cache_index(P, cblk, off, e), 8)) {
                        k[q] = load8<SRC>(P.src_k, sbase + e);
                        v[q] = load8<SRC>(P.src_v, sbase + e);
                    }
                }
                if (half == 0 && un < units) unit_index(nxt, node, blk);
                const float ks = CACHE && live && P.k_scale ? P.k_scale[si] : 1.f;
                const float vs = CACHE && live && P.v_scale ? P.v_scale[si] : 1.f;
#pragma unroll
                for (int q = 0; q < kV; ++q) {
                    const int e = e0 + (tid + (half * kV + q) * kThreads) * 8;
                    if (live && e < e1 &&
                        kv_index_ok(P, b, sbase + e, cache_index(P, cblk, off, e), 8)) {
                        const size_t di = cache_index(P, cblk, off, e);
                        store8<SRC, CACHE>(k[q], P.cache_k, di, ks);
                        store8<SRC, CACHE>(v[q], P.cache_v, di, vs);
                    }
                }
            }
        } else {
            if (un < units) unit_index(nxt, node, blk);
            const float ks = CACHE && live && P.k_scale ? P.k_scale[si] : 1.f;
            const float vs = CACHE && live && P.v_scale ? P.v_scale[si] : 1.f;
            for (int e = e0 + tid; live && e < e1; e += kThreads) {
                const size_t di = cache_index(P, cblk, off, e);
                if (!kv_index_ok(P, b, sbase + e, di, 1)) continue;
                put1<SRC, CACHE>(P.src_k, sbase + e, P.cache_k, di, ks);
                put1<SRC, CACHE>(P.src_v, sbase + e, P.cache_v, di, vs);
            }
        }
        u = un;
        cur = nxt;
    }
}

template <int SRC, int CACHE>
cudaError_t launch_kc(const KvCommitParams &p, bool vec, cudaStream_t st) {
    const int HD = p.H * p.D;
    const int pieces = (HD + kUnitElems - 1) / kUnitElems;
    const int64_t units = (int64_t)p.N * p.B * pieces;
    const int64_t cap = (int64_t)(p.sms > 0 ? p.sms : 1) * kCtasPerSm;
    const int grid = (int)(units < cap ? units : cap);
    const size_t smem = p.B <= kSmemRequests ? 2 * sizeof(int) * (size_t)p.B : 0;
    if (vec)
        kv_commit_kernel<SRC, CACHE, true><<<grid, kThreads, smem, st>>>(p, pieces);
    else
        kv_commit_kernel<SRC, CACHE, false><<<grid, kThreads, smem, st>>>(p, pieces);
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
