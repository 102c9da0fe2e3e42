"""Pins of the KV-commit oracle (CPU only): the fp8 encoder against torch's float8 conversion
(a library routine), a hand-worked placement in both cache layouts, and invariants."""
import numpy as np
import pytest
import torch

from oracle import kv_commit as K


@pytest.mark.parametrize("kind,tdtype,fmax", [(K.FP8_E4M3, torch.float8_e4m3fn, 448.0),
                                             (K.FP8_E5M2, torch.float8_e5m2, 57344.0)])
def test_fp8_encoder_matches_torch(kind, tdtype, fmax):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(800) * 1e-3,
                        rng.standard_normal(300) * 1e4,
                        [0.0, -0.0, 1e-12, -1e-12, fmax, -fmax, fmax * 1.01, 1e30]]).astype(np.float32)
    mine = K.fp8_encode(x, kind)
    ref = torch.from_numpy(np.clip(x, -fmax, fmax)).to(tdtype).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_fp8_saturates_and_keeps_sign_of_zero():
    e = K.fp8_encode(np.array([1e9, -1e9, -1e-30, 1e-30], np.float32), K.FP8_E4M3)
    assert e.tolist() == [0x7E, 0xFE, 0x80, 0x00]


def test_hand_worked_placement_both_layouts():
    """B=1, N=3 chain, accept_len 2 (root, node 1, node 2), block_size 2, blocks [3, 0],
    seq_pos 1: slot 0 -> p=1 -> block 3 offset 1; slot 1 -> p=2 -> block 0 offset 0;
    slot 2 -> p=3 -> block 0 offset 1."""
    H, D = 2, 3
    src_k = np.arange(3 * H * D, dtype=np.float32).reshape(1, 3, H, D)
    src_v = -src_k
    kv = np.array([[0, 1, 2]], np.int32)
    al = np.array([2], np.int32)
    table = np.array([[3, 0]], np.int32)
    pos = np.array([1], np.int32)
    for layout in (K.NHD, K.HND):
        shape = (4, 2, H, D) if layout == K.NHD else (4, H, 2, D)
        ck, cv, st = K.kv_commit(src_k, src_v, kv, al, np.full(shape, 99, np.float32),
                                 np.full(shape, 99, np.float32), layout, 2, table, pos)
        assert st.tolist() == [0]
        get = (lambda c, blk, off: c[blk, off]) if layout == K.NHD else \
            (lambda c, blk, off: c[blk, :, off])
        assert np.array_equal(get(ck, 3, 1), src_k[0, 0])
        assert np.array_equal(get(ck, 0, 0), src_k[0, 1])
        assert np.array_equal(get(ck, 0, 1), src_k[0, 2])
        assert np.array_equal(get(cv, 0, 1), src_v[0, 2])
        assert (get(ck, 3, 0) == 99).all() and (ck[1] == 99).all() and (ck[2] == 99).all()


def test_failed_request_and_bad_slot():
    H, D = 1, 2
    src = np.ones((2, 4, H, D), np.float32)
    kv = np.array([[-1, -1, -1, -1], [0, 2, 3, -1]], np.int32)
    al = np.array([0, 2], np.int32)
    table = np.array([[0, 1], [2, 3]], np.int32)
    pos = np.array([0, 2], np.int32)        # request 1: positions 2, 3, 4 -> block index 2 > table
    cache = np.zeros((4, 2, H, D), np.float32)
    ck, _, st = K.kv_commit(src, src, kv, al, cache, cache, K.NHD, 2, table, pos)
    assert st.tolist() == [0, K.BAD_SLOT]
    assert (ck[0] == 0).all() and (ck[1] == 0).all()          # request 0 wrote nothing
    assert (ck[3] == 1).all()                                    # positions 2, 3 -> block 3


def test_per_token_scales_hand_worked():
    """Per-token scales: slot j of the path divides by the scale of its source token (b, node).
    Chain 0 -> 1 -> 2 with K values 1.0, 3.0, 10.0 and per-node scales 0.5, 2.0, 4.0: the cache
    holds e4m3(2.0) = 0x40, e4m3(1.5) = 0x3C, e4m3(2.5) = 0x42 (bias 7: 2.0 = 2^1 -> 0x40,
    1.5 = 1.1b * 2^0 -> 0x3C, 2.5 = 1.01b * 2^1 -> 0x42); V with a scalar scale of 1 for
    comparison: 1.0 -> 0x38, 3.0 -> 0x44, 10.0 -> 0x52."""
    vals = np.array([1.0, 3.0, 10.0], np.float32).reshape(1, 3, 1, 1)
    kv = np.array([[0, 1, 2]], np.int32)
    al = np.array([2], np.int32)
    table = np.array([[0]], np.int32)
    pos = np.array([0], np.int32)
    cache = np.zeros((1, 4, 1, 1), np.uint8)
    ks = np.array([[0.5, 2.0, 4.0]], np.float32)
    ck, _, st = K.kv_commit(vals, vals, kv, al, cache, cache, K.NHD, 4, table, pos,
                            cache_kind=K.FP8_E4M3, k_scale=ks, v_scale=1.0)
    assert st.tolist() == [0]
    assert ck[0, :3, 0, 0].tolist() == [0x40, 0x3C, 0x42]
    _, cv, _ = K.kv_commit(vals, vals, kv, al, cache, cache, K.NHD, 4, table, pos,
                           cache_kind=K.FP8_E4M3, k_scale=ks, v_scale=1.0)
    assert cv[0, :3, 0, 0].tolist() == [0x38, 0x44, 0x52]


def test_uniform_per_token_scales_equal_the_scalar():
    rng = np.random.default_rng(3)
    B, N, H, D = 3, 5, 2, 4
    src = (rng.standard_normal((B, N, H, D)) * 5).astype(np.float32)
    kv = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    al = np.full(B, N - 1, np.int32)
    table = np.arange(B * 2, dtype=np.int32).reshape(B, 2)
    pos = np.zeros(B, np.int32)
    cache = np.zeros((B * 2, 4, H, D), np.uint8)
    a = K.kv_commit(src, src, kv, al, cache, cache, K.NHD, 4, table, pos, cache_kind=K.FP8_E5M2,
                    k_scale=0.75, v_scale=3.0)
    b = K.kv_commit(src, src, kv, al, cache, cache, K.NHD, 4, table, pos, cache_kind=K.FP8_E5M2,
                    k_scale=np.full((B, N), 0.75, np.float32),
                    v_scale=np.full((B, N), 3.0, np.float32))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
