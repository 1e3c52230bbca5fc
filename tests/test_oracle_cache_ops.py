"""Pins for the oracle's cache write (incl. FP8 quantisation) and block copy."""
import numpy as np
import pytest
import torch

from oracle.cache_ops import cache_write, copy_blocks, fp8_quantize_token
from oracle.fp8_e4m3 import e4m3_decode

BS = 16


def test_cache_write_places_rows_by_slot_and_skips_padding():
    rng = np.random.Generator(np.random.PCG64(1))
    nb, H, D = 5, 3, 8
    kc = rng.standard_normal((nb, H, BS, D)).astype(np.float16)
    vc = rng.standard_normal((nb, H, BS, D)).astype(np.float16)
    k = rng.standard_normal((4, H, D)).astype(np.float16)
    v = rng.standard_normal((4, H, D)).astype(np.float16)
    slots = np.array([17, -1, 79, 0])
    k2, v2, _, _ = cache_write(k, v, slots, kc, vc)
    # slot 17 -> block 1 row 1; 79 -> block 4 row 15; 0 -> block 0 row 0
    assert np.array_equal(k2[1, :, 1], k[0]) and np.array_equal(v2[1, :, 1], v[0])
    assert np.array_equal(k2[4, :, 15], k[2]) and np.array_equal(v2[4, :, 15], v[2])
    assert np.array_equal(k2[0, :, 0], k[3]) and np.array_equal(v2[0, :, 0], v[3])
    touched = np.zeros((nb, BS), bool)
    touched[1, 1] = touched[4, 15] = touched[0, 0] = True
    keep = ~np.broadcast_to(touched[:, None, :], (nb, H, BS))
    assert np.array_equal(k2[keep], kc[keep]) and np.array_equal(v2[keep], vc[keep])
    with pytest.raises(ValueError):
        cache_write(k, v, np.array([3, 3, -1, -1]), kc, vc)


def test_fp8_quantiser_properties():
    rng = np.random.Generator(np.random.PCG64(2))
    x = rng.standard_normal((8, 128)).astype(np.float32) * 3
    codes, scale = fp8_quantize_token(x)
    amax = np.abs(x).max()
    assert scale == np.float32(amax) / np.float32(448)
    # the largest-magnitude element lands on +-448 exactly
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert e4m3_decode(codes[i]) in (448.0, -448.0)
    # reconstruction within half a grid step (relative 2^-4) of every normal value
    rec = e4m3_decode(codes) * np.float64(scale)
    normal = np.abs(x / scale) >= 2.0 ** -6
    assert np.all(np.abs(rec - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 + 1e-12)
    # codes equal torch's float8 cast of the same float32 quotient
    ref = torch.from_numpy(x / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    # all-zero token: scale 1, zero codes
    c0, s0 = fp8_quantize_token(np.zeros((2, 4), np.float32))
    assert s0 == 1.0 and not c0.any()


def test_fp8_cache_write_stores_codes_and_per_token_scales():
    rng = np.random.Generator(np.random.PCG64(3))
    nb, H, D = 3, 2, 16
    kc = np.zeros((nb, H, BS, D), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((nb, BS), np.float32)
    vs = np.zeros_like(ks)
    k = rng.standard_normal((2, H, D)).astype(np.float16)
    v = rng.standard_normal((2, H, D)).astype(np.float16)
    k2, v2, ks2, vs2 = cache_write(k, v, np.array([5, 40]), kc, vc, ks, vs)
    for i, s in enumerate([5, 40]):
        c, sc = fp8_quantize_token(k[i].astype(np.float32))
        assert np.array_equal(k2[s // BS, :, s % BS], c) and ks2[s // BS, s % BS] == sc
        c, sc = fp8_quantize_token(v[i].astype(np.float32))
        assert np.array_equal(v2[s // BS, :, s % BS], c) and vs2[s // BS, s % BS] == sc
    assert ks2[0, 4] == 0 and not k2[0, :, 4].any()


def test_copy_blocks_copies_whole_blocks():
    rng = np.random.Generator(np.random.PCG64(4))
    kc = rng.standard_normal((6, 2, BS, 4))
    vc = rng.standard_normal((6, 2, BS, 4))
    ks = rng.standard_normal((6, BS)).astype(np.float32)
    vs = rng.standard_normal((6, BS)).astype(np.float32)
    k2, v2, ks2, vs2 = copy_blocks(kc, vc, [[0, 3], [5, 1]], ks, vs)
    assert np.array_equal(k2[3], kc[0]) and np.array_equal(v2[1], vc[5])
    assert np.array_equal(ks2[3], ks[0]) and np.array_equal(vs2[1], vs[5])
    for blk in (0, 2, 4, 5):
        assert np.array_equal(k2[blk], kc[blk]) and np.array_equal(v2[blk], vc[blk])
    with pytest.raises(ValueError):
        copy_blocks(kc, vc, [[0, 3], [3, 4]])
    with pytest.raises(ValueError):
        copy_blocks(kc, vc, [[0, 3], [1, 3]])


def test_swap_blocks_moves_blocks_between_pools():
    from oracle.cache_ops import swap_blocks
    rng = np.random.Generator(np.random.PCG64(9))
    gk, gv = rng.standard_normal((5, 2, BS, 4)), rng.standard_normal((5, 2, BS, 4))
    hk, hv = np.zeros((3, 2, BS, 4)), np.zeros((3, 2, BS, 4))
    hk2, hv2, _, _ = swap_blocks(hk, hv, gk, gv, [[4, 0], [1, 2]])
    assert np.array_equal(hk2[0], gk[4]) and np.array_equal(hv2[2], gv[1]) and not hk2[1].any()
    gk2, gv2, _, _ = swap_blocks(gk, gv, hk2, hv2, [[0, 3]])
    assert np.array_equal(gk2[3], gk[4]) and np.array_equal(gk2[0], gk[0])
    with pytest.raises(ValueError):
        swap_blocks(hk, hv, gk, gv, [[0, 1], [2, 1]])
