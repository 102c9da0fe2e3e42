"""spec_kv_commit against the KV-commit oracle through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

from oracle import kv_commit as K
from speculative_decoding_tree_mask_gb300 import binding as G
from speculative_decoding_tree_mask_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def h():
    G.load()
    with G.Handle(64, 64, 1 << 16, 0) as handle:
        yield handle


def _paths(rng, parent):
    """A random root path per request: (kv_commit, accept_len) as a verify call returns them."""
    B, N = parent.shape
    kv = np.full((B, N), -1, np.int32)
    al = np.zeros(B, np.int32)
    for b in range(B):
        node, path = 0, [0]
        while True:
            kids = [c for c in range(N) if c and parent[b, c] == node]
            if not kids or rng.random() < 0.25:
                break
            node = int(rng.choice(kids))
            path.append(node)
        kv[b, :len(path)] = path
        al[b] = len(path) - 1
    return kv, al


@pytest.mark.parametrize("src", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("cache", [K.SAME, K.FP8_E4M3, K.FP8_E5M2])
@pytest.mark.parametrize("layout", [K.NHD, K.HND])
@pytest.mark.parametrize("D", [128, 36])
@pytest.mark.parametrize("scales", ["tensor", "token"])
def test_kv_commit_matches_oracle(h, src, cache, layout, D, scales):
    if cache == K.SAME and scales == "token":
        pytest.skip("scales apply to fp8 caches only")
    rng = np.random.default_rng(hash((src, cache, layout, D, scales)) % 2**32)
    B, N, H, bs = 12, 16, 4, 16
    parent = np.stack([W.random_trie(rng, N, 6, 3) for _ in range(B)])
    kv, al = _paths(rng, parent)
    for b in (5, 7):                                # paths of at least 3 slots
        node, path = 0, [0]
        while len(path) < 3:
            kids = [c for c in range(N) if c and parent[b, c] == node]
            if not kids:
                break
            node = kids[0]
            path.append(node)
        kv[b] = -1
        kv[b, :len(path)] = path
        al[b] = len(path) - 1
        assert al[b] >= 2
    kv[3] = -1                                      # a failed request: nothing is written
    al[3] = 0
    max_blocks = 4
    num_blocks = B * max_blocks + 3
    table = rng.permutation(num_blocks)[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
    pos = rng.integers(0, max_blocks * bs - N, B).astype(np.int32)
    pos[5] = max_blocks * bs - 1                    # slots past the table: status 5
    table[7, 1] = num_blocks + 5                    # a block id outside the cache
    pos[7] = bs - 2
    kvals = (rng.standard_normal((B, N, H, D)) * 3).astype(np.float32)
    vvals = (rng.standard_normal((B, N, H, D)) * 3).astype(np.float32)
    tk = torch.from_numpy(kvals).to(TDT[src])
    tv = torch.from_numpy(vvals).to(TDT[src])
    kf, vf = tk.float().numpy(), tv.float().numpy()   # exact values of the source type
    shape = (num_blocks, bs, H, D) if layout == K.NHD else (num_blocks, H, bs, D)
    if scales == "tensor":
        ks, vs = 0.5, 2.0
    else:   # one scale per source token, [B, N]
        ks = (2.0 ** rng.uniform(-3, 3, (B, N))).astype(np.float32)
        vs = (2.0 ** rng.uniform(-3, 3, (B, N))).astype(np.float32)
    if cache == K.SAME:
        ck0 = torch.full(shape, -1024.0, dtype=TDT[src])
        cv0 = ck0.clone()
        ref_k, ref_v, ref_st = K.kv_commit(kf, vf, kv, al, ck0.float().numpy(),
                                           cv0.float().numpy(), layout, bs, table, pos)
    else:
        ck0 = torch.full(shape, 0x55, dtype=torch.uint8)
        cv0 = ck0.clone()
        ref_k, ref_v, ref_st = K.kv_commit(kf, vf, kv, al, ck0.numpy(), cv0.numpy(), layout, bs,
                                           table, pos, cache_kind=cache, k_scale=ks, v_scale=vs)
    gk, gv = ck0.to(DEV), cv0.to(DEV)
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    scale_k = torch.tensor(np.atleast_1d(ks), dtype=torch.float32, device=DEV)
    scale_v = torch.tensor(np.atleast_1d(vs), dtype=torch.float32, device=DEV)
    G.spec_kv_commit(h, tk.to(DEV), tv.to(DEV), torch.from_numpy(kv).to(DEV),
                     torch.from_numpy(al).to(DEV), gk, gv, layout,
                     torch.from_numpy(table).to(DEV), torch.from_numpy(pos).to(DEV),
                     cache_kind=cache, k_scale=scale_k if cache else None,
                     v_scale=scale_v if cache else None, commit_status=st)
    torch.cuda.synchronize()
    assert st.cpu().numpy().tolist() == ref_st.tolist()
    assert ref_st[5] == K.BAD_SLOT and ref_st[7] == K.BAD_SLOT
    if cache == K.SAME:
        assert np.array_equal(gk.cpu().float().numpy(), ref_k)
        assert np.array_equal(gv.cpu().float().numpy(), ref_v)
    else:
        assert np.array_equal(gk.cpu().numpy(), ref_k)
        assert np.array_equal(gv.cpu().numpy(), ref_v)


@pytest.mark.parametrize("cache", [K.FP8_E4M3, K.FP8_E5M2])
def test_kv_commit_fp8_quotients_at_rounding_boundaries(h, cache):
    """The fp8 encoding of x / scale near every fp8 rounding boundary: quotients placed on the
    midpoints between adjacent fp8 values (ties to even), up to six float32 steps either side
    of them (the library's shortcut defers within three), beyond the largest finite value (saturation) and under the smallest subnormal (zero),
    for scales that are powers of two (the quotients land on the midpoints exactly) and scales
    that are not. These are the cases where the library's reciprocal shortcut must defer to the
    correctly rounded division; the cache must equal the oracle's encoding bit for bit."""
    rng = np.random.default_rng(90 + cache)
    vals = K._fp8_table(cache)[:0x7F]
    vals = np.sort(vals[np.isfinite(vals)])
    mids = (vals[1:] + vals[:-1]) / 2
    mids = np.concatenate([mids, [vals[-1] * 1.0625, vals[-1] * 4.0]])      # saturation
    least = vals[vals > 0][0]          # quotients under the smallest subnormal, down to zero
    mids = np.concatenate([mids, least * np.array([0.3, 0.2, 0.126, 0.124, 0.1, 1e-3]),
                           [1e-30, 1e-40]])
    t = mids.astype(np.float32)
    steps = (t.view(np.int32)[:, None] + np.arange(-6, 7, dtype=np.int32)[None, :]).ravel()
    t = steps.astype(np.int32).view(np.float32)
    t = np.concatenate([t, -t, np.float32([0.0, -0.0])])   # and zeros of both signs
    B, N, H, D = 4, 8, 2, 64
    per = H * D
    slots = B * N
    total = slots * per
    t = np.resize(rng.permutation(t), total).astype(np.float32)
    scale = (2.0 ** rng.uniform(-4, 4, (B, N)) * rng.uniform(1.01, 1.99, (B, N))).astype(
        np.float32)
    scale[:, ::2] = 2.0 ** rng.integers(-4, 5, (B, N // 2))   # powers of two: exact ties
    x = (t.reshape(B, N, H, D) * scale[:, :, None, None]).astype(np.float32)
    kv = np.tile(np.arange(N, dtype=np.int32), (B, 1))        # every node committed
    al = np.full(B, N - 1, np.int32)
    bs, max_blocks = 8, 1
    table = np.arange(B, dtype=np.int32).reshape(B, 1)
    pos = np.zeros(B, np.int32)
    shape = (B, bs, H, D)
    ck0 = torch.zeros(shape, dtype=torch.uint8)
    ref_k, ref_v, ref_st = K.kv_commit(x, x, kv, al, ck0.numpy(), ck0.numpy(), K.NHD, bs, table,
                                       pos, cache_kind=cache, k_scale=scale, v_scale=scale)
    gk, gv = ck0.to(DEV), ck0.clone().to(DEV)
    tx = torch.from_numpy(x).to(DEV)
    st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    sc = torch.from_numpy(scale).to(DEV)
    G.spec_kv_commit(h, tx, tx, torch.from_numpy(kv).to(DEV), torch.from_numpy(al).to(DEV), gk,
                     gv, K.NHD, torch.from_numpy(table).to(DEV), torch.from_numpy(pos).to(DEV),
                     cache_kind=cache, k_scale=sc, v_scale=sc, commit_status=st)
    torch.cuda.synchronize()
    assert st.cpu().numpy().tolist() == ref_st.tolist() == [0] * B
    assert np.array_equal(gk.cpu().numpy(), ref_k)
    assert np.array_equal(gv.cpu().numpy(), ref_v)


@pytest.mark.parametrize("cache,scale", [(K.SAME, None), (K.FP8_E4M3, 0.25),
                                         (K.FP8_E5M2, 0.0173)])
@pytest.mark.parametrize("B,H,D", [(1030, 2, 16), (4, 33, 128)])
def test_kv_commit_many_requests_and_pieces(cache, scale, B, H, D):
    """More requests than a CTA keeps in shared memory (1030 > 1024: the accepted length and
    position of each unit's request are read from global memory instead), and slots of
    33 x 128 = 4224 elements (two units each, 4096 + 128)."""
    rng = np.random.default_rng(B + 7 * cache)
    N, bs = 4, 8
    al = rng.integers(0, N, B).astype(np.int32)           # chains: slots 0..al[b]
    kv = np.full((B, N), -1, np.int32)
    for b in range(B):
        kv[b, :al[b] + 1] = np.arange(al[b] + 1)
    kv[B // 2] = -1                                       # a failed request
    al[B // 2] = 0
    table = rng.permutation(B).reshape(B, 1).astype(np.int32)
    pos = rng.integers(0, bs - N + 1, B).astype(np.int32)
    src = torch.from_numpy((rng.standard_normal((B, N, H, D)) * 2).astype(np.float32))
    tk, tv = src.to(torch.bfloat16), (src * -0.5).to(torch.bfloat16)
    kf, vf = tk.float().numpy(), tv.float().numpy()
    shape = (B, bs, H, D)
    if cache == K.SAME:
        ck0 = torch.full(shape, 3.0, dtype=torch.bfloat16)
        ref_k, ref_v, ref_st = K.kv_commit(kf, vf, kv, al, ck0.float().numpy(),
                                           ck0.float().numpy(), K.NHD, bs, table, pos)
    else:
        ck0 = torch.full(shape, 0x33, dtype=torch.uint8)
        ref_k, ref_v, ref_st = K.kv_commit(kf, vf, kv, al, ck0.numpy(), ck0.numpy(), K.NHD, bs,
                                           table, pos, cache_kind=cache, k_scale=scale,
                                           v_scale=scale)
    with G.Handle(B, N, 1 << 10, 0) as hh:
        gk, gv = ck0.to(DEV), ck0.clone().to(DEV)
        st = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        sc = torch.tensor([scale], dtype=torch.float32, device=DEV) if scale else None
        G.spec_kv_commit(hh, tk.to(DEV), tv.to(DEV), torch.from_numpy(kv).to(DEV),
                         torch.from_numpy(al).to(DEV), gk, gv, K.NHD,
                         torch.from_numpy(table).to(DEV), torch.from_numpy(pos).to(DEV),
                         cache_kind=cache, k_scale=sc, v_scale=sc, commit_status=st)
        torch.cuda.synchronize()
    assert st.cpu().numpy().tolist() == ref_st.tolist() == [0] * B
    got_k = gk.cpu().float().numpy() if cache == K.SAME else gk.cpu().numpy()
    got_v = gv.cpu().float().numpy() if cache == K.SAME else gv.cpu().numpy()
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_v, ref_v)
