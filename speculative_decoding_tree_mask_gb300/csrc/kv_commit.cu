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
// fp8 caches hold the fp8 rounding (nearest, ties to even, saturated, the sign kept also when
// the magnitude rounds to zero) of x / scale rounded to float32 first; the scale is one value
// per tensor or one per source token (b, node).
//
// Work is split into units of (slot j, request b, piece of 4096 of the slot's H*D elements),
// ordered slot-major, so that the slots every request commits (j <= accept_len) come first.
// A grid of one wave of CTAs (the occupancy query decides: 8 to 10 per SM, registers bound it)
// strides over the units. Each CTA first reads every request's accepted length and position
// into shared memory and stops at the deepest accepted slot of the batch, so no CTA works on a
// slot nobody commits; the node of its first unit is loaded in the same round trip. The copy
// is staged through shared memory with cp.async: each thread copies its own 16-byte vectors of
// the unit's K and V rows there, waits for its own copies (cp.async.wait_group: a hardware wait
// on the thread's own group, no spinning) and stores them to the cache, so the data occupies
// no registers (holding it in registers allowed 6 CTAs per SM). A unit costs two round trips:
// its node (loaded with the previous unit's data) starts the copies, and its cache block is
// loaded while they are in flight. The statuses are checked by the CTAs that get the fewest
// units.

#include <cfloat>
#include <cuda_fp16.h>

#include "spec_device.cuh"
#include "spec_internal.h"

namespace specv {
namespace {

constexpr int kThreads = 128;
constexpr int kVecs = 4;                          // 8-element vectors per thread per unit
constexpr int kUnitElems = kThreads * 8 * kVecs;  // elements of K (and of V) per unit
constexpr int kCtasPerSm = 12;   // at most (16 KiB of staging per CTA for 16-bit sources)
constexpr int kSmemRequests = 1024;               // requests whose (L, position) fit in smem

template <int SRC>
constexpr int src_bytes() { return SRC == 0 ? 4 : 2; }

template <int SRC>
__device__ __forceinline__ float src_elem(const void *p, size_t i) {
    if (SRC == 0) return __ldg(reinterpret_cast<const float *>(p) + i);
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
    if (SRC == 1) return __uint_as_float(uint32_t(h) << 16);
    return __half2float(__ushort_as_half(h));
}

// Two fp8 codes: code(a) in the low byte, code(b) in the high byte (nearest, ties to even,
// saturated at the largest finite value).
__device__ __forceinline__ uint16_t fp8x2(float a, float b, int kind) {
    uint16_t r;
    if (kind == 1)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
    return r;
}

// fp8 code of a float (nearest, ties to even, saturated; sign-magnitude, so a negative value
// that rounds to zero is -0: the conversion instruction returns +0 there, so the magnitude is
// converted and the sign set apart); NaN gives 0x7F.
template <int CACHE>
__device__ __forceinline__ uint32_t fp8_of(float q) {
    if (q != q) return 0x7fu;
    return (fp8x2(fabsf(q), 0.f, CACHE) & 0xffu) | ((__float_as_uint(q) >> 24) & 0x80u);
}

// The float32 quotient RN(x / s) for the fp8 encoding, given y = RN(1 / s) for a scale s whose
// reciprocal is a normal float, without a division. q0 = RN(x y) is within about one ulp of
// x / s, and one correction with the residual (two fused multiply-adds) leaves q1 within about
// half an ulp, so RN(x / s) lies within two representable steps of q1. The fp8 code of a value
// changes only where the value crosses a rounding boundary, a midpoint between two adjacent fp8
// values. fp8 values are the multiples of 2^(E - KB) in binade E >= Emin (KB mantissa bits) and
// the multiples of 2^(Emin - KB) below 2^Emin (the subnormals), so in q1's binade e the
// midpoints are the values whose low 23 - k mantissa bits are exactly 100...0, with
// k = KB - max(Emin - e, 0) bits kept. When q1's low bits lie more than two steps from that
// pattern, q1 and RN(x / s) encode alike and q1 is returned with `ok` set; so it is when the
// residual x - q1 s is exactly zero (q1 is then the exact quotient: a power-of-two scale, or a
// 16-bit source value that sits on a midpoint itself). Magnitudes beyond
// Emax saturate to the largest finite value, and those below a quarter of the smallest
// subnormal round to zero, either way. Anything else (two steps from a midpoint, the binades
// just under the smallest subnormal, a non-finite value) clears `ok`, and the caller takes the
// correctly rounded division. The sign is that of x times s (the correction step can turn -0
// into +0).
template <int CACHE>
__device__ __forceinline__ float fp8_quotient(float x, float s, float y, bool &ok) {
    constexpr int KB = CACHE == 1 ? 3 : 2;           // mantissa bits kept by fp8 normals
    constexpr int EMIN = CACHE == 1 ? -6 : -14;      // fp8 normal binades [EMIN, EMAX]
    constexpr int EMAX = CACHE == 1 ? 8 : 15;
    const float q0 = x * y;
    const float q1 = fmaf(fmaf(-q0, s, x), y, q0);
    const uint32_t mag = __float_as_uint(q1) & 0x7fffffffu;
    const int e = (int)(mag >> 23) - 127;
    const int k = KB - max(EMIN - e, 0);             // >= 0 for e >= EMIN - KB
    const uint32_t half = 1u << (22 - max(k, 0));
    const uint32_t low = mag & (2u * half - 1u);
    ok = mag < 0x7f800000u &&
         (e > EMAX || e < EMIN - KB - 2 || (k >= 0 && (low + 2u < half || low > half + 2u)) ||
          fmaf(-q1, s, x) == 0.f);
    const uint32_t sign = (__float_as_uint(x) ^ __float_as_uint(s)) & 0x80000000u;
    return __uint_as_float(mag | sign);
}

// The correctly rounded division, kept out of line: it runs for a few elements in a million.
__device__ __noinline__ float div_rn(float x, float s) { return __fdiv_rn(x, s); }

// The common case, cheaper still: q0 = RN(x y) alone. With y = RN(1/s), x y = (x/s)(1 + e1)
// and q0 = x y (1 + e2), |e1|, |e2| <= 2^-24, so q0 is within 2^-23 |x/s|, two steps of its own
// binade, of x / s, and RN(x / s) within half a step more: within three steps of q0. So q0 in
// the fp8 normal binades with its dropped mantissa bits more than three steps from the
// midpoint pattern encodes like RN(x / s). Elements that fail this test take
// fp8_quotient_full (zeros, the subnormal range, saturation, near-ties, exact quotients,
// non-finite). Power-of-two scales, whose quotients are exact and land on fp8 midpoints often
// (one 16-bit source value in 16 for e4m3), never come here.
template <int CACHE>
__device__ __forceinline__ float fp8_q0(float x, float y) {
    return x * y;
}
template <int CACHE>
__device__ __forceinline__ bool fp8_fast_ok(float q0) {
    constexpr int KB = CACHE == 1 ? 3 : 2;
    constexpr int EMIN = CACHE == 1 ? -6 : -14;
    constexpr int EMAX = CACHE == 1 ? 8 : 15;
    constexpr uint32_t LO = uint32_t(127 + EMIN) << 23, RANGE = uint32_t(EMAX - EMIN + 1) << 23;
    constexpr uint32_t DROP = (1u << (23 - KB)) - 1u, HALF = 1u << (22 - KB);
    const uint32_t mag = __float_as_uint(q0) & 0x7fffffffu;
    return mag - LO < RANGE && (mag & DROP) - HALF + 3u > 6u;
}
template <int CACHE>
__device__ __noinline__ float fp8_quotient_full(float x, float s, float y, bool fast) {
    bool ok = false;
    const float q = fast ? fp8_quotient<CACHE>(x, s, y, ok) : 0.f;
    return ok ? q : div_rn(x, s);
}

// How a scale's quotients are formed: a power-of-two scale (its reciprocal exact, so
// x * RN(1/s) is the same real number as x / s and rounds alike: one multiply, no test), a
// scale with a normal reciprocal (fp8_q0 and fp8_fast_ok, then fp8_quotient_full), or the
// correctly rounded division for every element.
enum { Q_POW2 = 0, Q_RECIP = 1, Q_DIV = 2 };
__device__ __forceinline__ int scale_mode(float s) {
    const uint32_t u = __float_as_uint(s) & 0x7fffffffu;
    if ((u & 0x7fffffu) == 0u && u >= 0x00800000u && u <= 0x7e800000u) return Q_POW2;
    const float a = fabsf(s);
    return a >= 1e-37f && a <= 1e37f ? Q_RECIP : Q_DIV;
}

// One element src[si] -> cache[di] (the unvectorised path).
template <int SRC, int CACHE>
__device__ __forceinline__ void put1(const void *src, size_t si, void *dst, size_t di,
                                     float scale, float rcp, int mode) {
    if (CACHE == 0) {
        if (SRC == 0)
            reinterpret_cast<float *>(dst)[di] = __ldg(reinterpret_cast<const float *>(src) + si);
        else
            reinterpret_cast<unsigned short *>(dst)[di] =
                __ldg(reinterpret_cast<const unsigned short *>(src) + si);
    } else {
        const float x = src_elem<SRC>(src, si);
        reinterpret_cast<uint8_t *>(dst)[di] = (uint8_t)fp8_of<CACHE>(
            mode == Q_POW2 ? x * rcp : fp8_quotient_full<CACHE>(x, scale, rcp, mode == Q_RECIP));
    }
}

// 16-byte asynchronous copy global -> shared (bypassing L1), and the waits on this thread's
// copies.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Store one staged 8-element vector (`raw`: one 16-byte word for 16-bit sources, two for f32)
// at cache element di.
template <int SRC, int CACHE>
__device__ __forceinline__ void store8(const uint4 *raw, void *dst, size_t di, float scale,
                                       float rcp, int mode) {
    if (CACHE == 0) {
        uint4 *dp = reinterpret_cast<uint4 *>(reinterpret_cast<char *>(dst) +
                                              di * (size_t)src_bytes<SRC>());
        dp[0] = raw[0];
        if (SRC == 0) dp[1] = raw[1];
        return;
    }
    float x[8];
    if (SRC == 0) {
        const uint4 a = raw[0], b = raw[1];
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
        x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    } else {
        const uint4 a = raw[0];
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
    float q[8];
    // clean: every quotient is finite and at least the smallest fp8 subnormal in magnitude, so
    // its code is nonzero, the conversion keeps its sign, and no NaN or -0 needs fixing
    bool clean = false;
    if (mode == Q_POW2) {
        constexpr uint32_t LEAST = uint32_t(127 + (CACHE == 1 ? -9 : -16)) << 23;
        unsigned odd = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[i] = x[i] * rcp;
            odd |= (__float_as_uint(q[i]) & 0x7fffffffu) - LEAST >= 0x7f800000u - LEAST;
        }
        clean = odd == 0u;
    } else {
        unsigned slow = mode == Q_RECIP ? 0u : 0xffu;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q[i] = fp8_q0<CACHE>(x[i], rcp);
            slow |= fp8_fast_ok<CACHE>(q[i]) ? 0u : 1u << i;
        }
        if (slow) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (slow & (1u << i))
                    q[i] = fp8_quotient_full<CACHE>(x[i], scale, rcp, mode == Q_RECIP);
        }
        clean = slow == 0u;
    }
    // pairs (one conversion per two elements); unless clean, the signs OR'd in (the conversion
    // gives +0 for a negative value that rounds to zero, the format keeps -0) and NaN as 0x7F
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = fp8x2(q[2 * i], q[2 * i + 1], CACHE);
    if (!clean) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c[i] |= ((__float_as_uint(q[2 * i]) >> 24) & 0x80u) |
                    ((__float_as_uint(q[2 * i + 1]) >> 16) & 0x8000u);
            if (q[2 * i] != q[2 * i]) c[i] = (c[i] & 0xff00u) | 0x7fu;
            if (q[2 * i + 1] != q[2 * i + 1]) c[i] = (c[i] & 0x00ffu) | 0x7f00u;
        }
    }
    uint2 o;
    o.x = c[0] | (c[1] << 16);
    o.y = c[2] | (c[3] << 16);
    *reinterpret_cast<uint2 *>(reinterpret_cast<char *>(dst) + di) = o;
}

// Cache element of (slot position `off` in block `blk`, element e of the H*D slot). In the
// NHD layout a slot's H*D elements are contiguous, so no division is needed there.
__device__ __forceinline__ size_t cache_index(const KvCommitParams &P, int blk, int off, int e) {
    if (P.layout == 0) return ((size_t)blk * P.block_size + off) * ((size_t)P.H * P.D) + e;
    const int h = e / P.D, d = e - h * P.D;
    return (((size_t)blk * P.H + h) * P.block_size + off) * (size_t)P.D + d;
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

// One unit of work: slot j of request b, piece `piece` of the slot's H*D elements.
struct Unit {
    int j, b, piece, L, pos;
};

template <int SRC, int CACHE, bool VEC>
__global__ void __launch_bounds__(kThreads, 8)
    kv_commit_kernel(KvCommitParams P, int pieces, int cached) {
    // dynamic shared memory: [staging: K then V rows of one unit][2][B] (last slot, position)
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRowBytes = kUnitElems * src_bytes<SRC>();
    uint4 *stage_k = reinterpret_cast<uint4 *>(smem);
    uint4 *stage_v = reinterpret_cast<uint4 *>(smem + kRowBytes);
    int *s_req = reinterpret_cast<int *>(smem + (VEC ? 2 * kRowBytes : 0));
    __shared__ int s_max;
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = P.B, N = P.N, G = (int)gridDim.x;
    const int64_t per_slot = (int64_t)B * pieces;
    // 32-bit division when the unit indices fit (they do for any batch with N*B*pieces < 2^31)
    const bool small = (int64_t)N * per_slot < (int64_t(1) << 31);
    auto decode = [&](int64_t u, Unit &x) {
        if (small) {
            const uint32_t u32 = (uint32_t)u, ps = (uint32_t)per_slot;
            x.j = (int)(u32 / ps);
            const uint32_t r = u32 - (uint32_t)x.j * ps;
            x.b = (int)(r / (uint32_t)pieces);
            x.piece = (int)(r - (uint32_t)x.b * (uint32_t)pieces);
            return;
        }
        x.j = (int)(u / per_slot);
        const int64_t r = u - (int64_t)x.j * per_slot;
        x.b = (int)(r / pieces);
        x.piece = (int)(r - (int64_t)x.b * pieces);
    };
    // The first unit's node is loaded with the prologue, before its liveness is known (any
    // unit index names a valid kv_commit entry).
    Unit first;
    decode(blockIdx.x, first);
    const int first_node = __ldg(P.kv_commit + (size_t)first.b * N + first.j);
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
    const int64_t units = (int64_t)(max(lmax, 0) + 1) * per_slot;
    // The CTA's next unit at or after u (stride G) that copies something; units when none.
    auto next_live = [&](int64_t u, Unit &x) -> int64_t {
        for (; u < units; u += G) {
            decode(u, x);
            x.L = cached ? s_req[x.b] : last_slot(P, x.b);
            if (x.j > x.L) continue;   // failed verification, or a slot it does not commit
            x.pos = cached ? s_req[B + x.b] : P.seq_pos[x.b];
            return u;
        }
        return units;
    };

    Unit cur;
    int64_t u = next_live(blockIdx.x, cur);
    int node = u == (int64_t)blockIdx.x ? first_node
                                        : (u < units ? __ldg(P.kv_commit + (size_t)cur.b * N +
                                                             cur.j)
                                                     : -1);
    while (u < units) {
        const int b = cur.b;
        const int p = cur.pos + cur.j;
        const bool src_ok = node >= 0 && node < N;
        const size_t sbase = ((size_t)b * N + (src_ok ? node : 0)) * (size_t)HD;
        const int e0 = cur.piece * kUnitElems, e1 = min(HD, e0 + kUnitElems);
        if (VEC && src_ok) {
            // this thread's vectors of the unit's K and V rows -> its own staging slots
#pragma unroll
            for (int q = 0; q < kVecs; ++q) {
                const int e = e0 + (tid + q * kThreads) * 8;
                if (e < e1) {
                    const char *sk = reinterpret_cast<const char *>(P.src_k) +
                                     (sbase + e) * (size_t)src_bytes<SRC>();
                    const char *sv = reinterpret_cast<const char *>(P.src_v) +
                                     (sbase + e) * (size_t)src_bytes<SRC>();
                    const int sl = (tid + q * kThreads) * (SRC == 0 ? 2 : 1);
                    cp_async16(stage_k + sl, sk);
                    cp_async16(stage_v + sl, sv);
                    if (SRC == 0) {
                        cp_async16(stage_k + sl + 1, sk + 16);
                        cp_async16(stage_v + sl + 1, sv + 16);
                    }
                }
            }
            cp_async_commit();
        }
        // the cache block and the scales, while the copies are in flight
        const int bi = p >= 0 ? p / P.block_size : -1;
        const int blk = (bi >= 0 && bi < P.max_blocks)
                            ? __ldg(P.block_table + (size_t)b * P.max_blocks + bi)
                            : -1;
        const size_t si = P.scale_per_token ? (size_t)b * N + (src_ok ? node : 0) : 0;
        const float ks = CACHE && P.k_scale ? P.k_scale[si] : 1.f;
        const float vs = CACHE && P.v_scale ? P.v_scale[si] : 1.f;
        // the next unit's node
        Unit nxt;
        const int64_t un = next_live(u + G, nxt);
        const int nnode = un < units ? __ldg(P.kv_commit + (size_t)nxt.b * N + nxt.j) : -1;
        const bool live = src_ok && blk >= 0 && blk < P.num_blocks;
        const int off = live ? p - bi * P.block_size : 0;
        const int kmode = CACHE ? scale_mode(ks) : Q_DIV, vmode = CACHE ? scale_mode(vs) : Q_DIV;
        const float krcp = kmode != Q_DIV ? __frcp_rn(ks) : 1.f;
        const float vrcp = vmode != Q_DIV ? __frcp_rn(vs) : 1.f;
        if (VEC) {
            if (src_ok) cp_async_wait_all();   // this thread's own copies
#pragma unroll
            for (int q = 0; q < kVecs; ++q) {
                const int e = e0 + (tid + q * kThreads) * 8;
                if (live && e < e1 &&
                    kv_index_ok(P, b, sbase + e, cache_index(P, blk, off, e), 8)) {
                    const size_t di = cache_index(P, blk, off, e);
                    const int sl = (tid + q * kThreads) * (SRC == 0 ? 2 : 1);
                    store8<SRC, CACHE>(stage_k + sl, P.cache_k, di, ks, krcp, kmode);
                    store8<SRC, CACHE>(stage_v + sl, P.cache_v, di, vs, vrcp, vmode);
                }
            }
        } else {
            for (int e = e0 + tid; live && e < e1; e += kThreads) {
                const size_t di = cache_index(P, blk, off, e);
                if (!kv_index_ok(P, b, sbase + e, di, 1)) continue;
                put1<SRC, CACHE>(P.src_k, sbase + e, P.cache_k, di, ks, krcp, kmode);
                put1<SRC, CACHE>(P.src_v, sbase + e, P.cache_v, di, vs, vrcp, vmode);
            }
        }
        u = un;
        cur = nxt;
        node = nnode;
    }
}

template <int SRC, int CACHE>
cudaError_t launch_kc(const KvCommitParams &p, bool vec, cudaStream_t st) {
    const int HD = p.H * p.D;
    const int pieces = (HD + kUnitElems - 1) / kUnitElems;
    const int64_t units = (int64_t)p.N * p.B * pieces;
    const int cached = p.B <= kSmemRequests;
    const size_t stage = vec ? 2 * (size_t)kUnitElems * src_bytes<SRC>() : 0;
    const size_t smem = stage + (cached ? 2 * sizeof(int) * (size_t)p.B : 0);
    auto kernel = vec ? kv_commit_kernel<SRC, CACHE, true> : kv_commit_kernel<SRC, CACHE, false>;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // CTAs resident per SM (12 with 16 KiB of staging; fewer for f32 sources): the grid is one
    // wave of them at most
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    per_sm = per_sm < kCtasPerSm ? per_sm : kCtasPerSm;
    const int64_t cap = (int64_t)(p.sms > 0 ? p.sms : 1) * per_sm;
    const int grid = (int)(units < cap ? units : cap);
    kernel<<<grid, kThreads, smem, st>>>(p, pieces, cached);
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
