"""Oracle of the KV commit that follows verification (numpy, written from the definitions).

TEST INFRASTRUCTURE: used by the test suite only; shares no code with the CUDA path.

IluvatarLabs/vllm PR #3 ("SCV vectorized masking", commit implementing `commit_draft_kernel`)
copies the K/V of accepted draft tokens into the paged KV cache: NHD or HND cache layouts,
fp16/bf16/fp32 sources, a cache of the source type or fp8 (e4m3 / e5m2) with a scale, and an
early return for masked (rejected) entries. EmbodiInfer PR #11 (commits 938fe7b
"incremental_kv_commit" and 41dcd00 "compacts the pooled KV in batches") commits only the new
tokens of a turn. Here, for request b the slots j = 0..accept_len[b] of kv_commit[b] (the root,
then the accepted nodes in path order) are written at sequence positions seq_pos[b] + j:
    block = block_table[b][p // block_size], offset = p % block_size,
    NHD cache [num_blocks, block_size, H, D], HND cache [num_blocks, H, block_size, D].
fp8 caches store fp8(x / scale) with x / scale rounded to float32 first, then rounded to the
nearest fp8 value (ties to the even code) and saturated to the largest finite value. The
commit kernel takes a scalar scale or one scale per token: a scale given as a [B, N] array is
the scale of source token (b, node).
A request whose kv_commit[b][0] < 0 (verification failed) writes nothing; a slot whose block
lies outside the table or the cache writes nothing and sets commit_status[b] = 5.
"""
from __future__ import annotations

import numpy as np

NHD, HND = 0, 1
F32, BF16, F16 = 0, 1, 2
SAME, FP8_E4M3, FP8_E5M2 = 0, 1, 2
BAD_SLOT = 5


def _fp8_table(kind: int) -> np.ndarray:
    """Values of all 256 fp8 codes (float64; NaN codes as NaN)."""
    vals = np.empty(256)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        if kind == FP8_E4M3:
            e, m = (code >> 3) & 0xF, code & 0x7
            if e == 0xF and m == 0x7:
                vals[code] = np.nan
            elif e == 0:
                vals[code] = s * (m / 8.0) * 2.0 ** (1 - 7)
            else:
                vals[code] = s * (1 + m / 8.0) * 2.0 ** (e - 7)
        else:
            e, m = (code >> 2) & 0x1F, code & 0x3
            if e == 0x1F:
                vals[code] = np.nan if m else s * np.inf
            elif e == 0:
                vals[code] = s * (m / 4.0) * 2.0 ** (1 - 15)
            else:
                vals[code] = s * (1 + m / 4.0) * 2.0 ** (e - 15)
    return vals


_TABLES = {}


def fp8_encode(x: np.ndarray, kind: int) -> np.ndarray:
    """Round float32 values to the nearest finite fp8 value, ties to the even code, saturating
    at the largest finite magnitude; the sign is carried separately (sign-magnitude format),
    so a negative value that rounds to zero gives -0."""
    if kind not in _TABLES:
        _TABLES[kind] = _fp8_table(kind)
    vals = _TABLES[kind]
    mags = np.arange(0x80)                           # non-negative codes
    fv = vals[mags]
    ok = np.isfinite(fv)
    mags, fv = mags[ok], fv[ok]
    maxf = np.max(fv)
    x = np.asarray(x, dtype=np.float64).ravel()
    out = np.empty(x.shape, np.uint8)
    for i, v in enumerate(x):
        if np.isnan(v):
            out[i] = 0x7F
            continue
        a = min(abs(v), maxf)
        d = np.abs(fv - a)
        cand = mags[d == np.min(d)]
        code = int(cand[0]) if len(cand) == 1 else int(next(c for c in cand if c % 2 == 0))
        out[i] = code | (0x80 if np.signbit(v) else 0)
    return out


def kv_commit(src_k, src_v, kv_commit_idx, accept_len, cache_k, cache_v, layout, block_size,
              block_table, seq_pos, cache_kind=SAME, k_scale=1.0, v_scale=1.0):
    """src_k/src_v: [B, N, H, D] (float32, or uint16 bf16/f16 bit patterns are NOT accepted:
    pass float32 values and the cache's element view). Returns (cache_k, cache_v, status)
    updated copies. Caches are numpy arrays of the stored element type (float32 / uint16 for
    16-bit types / uint8 for fp8)."""
    B, N, H, D = src_k.shape
    ck, cv = cache_k.copy(), cache_v.copy()
    num_blocks = ck.shape[0]
    status = np.zeros(B, np.int32)
    for b in range(B):
        if kv_commit_idx[b, 0] < 0:
            continue
        for j in range(int(accept_len[b]) + 1):
            node = int(kv_commit_idx[b, j])
            p = int(seq_pos[b]) + j
            bi = p // block_size
            if p < 0 or bi >= block_table.shape[1]:
                status[b] = BAD_SLOT
                continue
            blk = int(block_table[b, bi])
            if blk < 0 or blk >= num_blocks:
                status[b] = BAD_SLOT
                continue
            off = p % block_size
            for cache, src, scale in ((ck, src_k, k_scale), (cv, src_v, v_scale)):
                x = src[b, node]                          # [H, D] float32 values
                if cache_kind == SAME:
                    val = x
                else:
                    s = scale[b, node] if np.ndim(scale) == 2 else scale
                    q = (x.astype(np.float32) / np.float32(s)).astype(np.float32)
                    val = fp8_encode(q, cache_kind).reshape(H, D)
                if layout == NHD:
                    cache[blk, off] = val
                else:
                    cache[blk, :, off] = val
    return ck, cv, status
