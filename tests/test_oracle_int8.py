"""Pins for the oracle's INT8 KV format (per-token symmetric scale).

The reading: scale = fl32(amax / 127) (1 for an all-zero token), code =
round-half-even(fl32(x / scale)) in [-127, 127], stored value code * scale.
Pinned by closed forms: a token whose amax is 127 has scale exactly 1, so its
codes are the round-half-even integers of the inputs (ties checked at every
half-integer of a range); the amax element maps to +-127; every element is
reconstructed within half a step; an all-zero token has scale 1 and zero
codes; the cache write dispatches on the cache dtype; and attention over an
INT8 cache equals attention over the same values stored as floats.
"""
import numpy as np

from oracle.attention import paged_decode
from oracle.cache_ops import int8_quantize_rows, fp8_quantize_rows, cache_write


def test_ties_round_to_even_at_unit_scale():
    halves = np.arange(-126.5, 127.0, 1.0, dtype=np.float32)          # every half-integer
    x = np.concatenate([[127.0], halves]).astype(np.float32)[None]      # amax 127 -> scale 1
    codes, scale = int8_quantize_rows(x)
    assert scale[0] == np.float32(1.0)
    evens = np.where(np.floor(halves) % 2 == 0, np.floor(halves), np.ceil(halves))
    assert codes[0, 0] == 127
    assert np.array_equal(codes[0, 1:].astype(np.int64), evens.astype(np.int64))


def test_amax_maps_to_127_and_reconstruction_is_within_half_a_step():
    rng = np.random.Generator(np.random.PCG64(3))
    x = (rng.standard_normal((500, 2, 64)) * rng.uniform(1e-3, 1e3, size=(500, 1, 1))).astype(np.float32)
    codes, scale = int8_quantize_rows(x)
    flat = x.reshape(500, -1)
    c = codes.reshape(500, -1).astype(np.int64)
    arg = np.abs(flat).argmax(axis=1)
    assert np.array_equal(np.abs(c[np.arange(500), arg]), np.full(500, 127))
    assert np.all(np.abs(c) <= 127)
    err = np.abs(c * scale[:, None].astype(np.float64) - flat.astype(np.float64))
    assert np.all(err <= 0.5 * scale[:, None] * (1 + 1e-6))
    # the scale is amax / 127 rounded to float32
    amax = np.abs(flat).max(axis=1)
    assert np.all(np.abs(scale.astype(np.float64) * 127 - amax) <= amax * 2.0 ** -23 * 127)


def test_zero_token():
    codes, scale = int8_quantize_rows(np.zeros((1, 3, 8), np.float32))
    assert scale[0] == 1.0 and not codes.any()


def test_cache_write_dispatches_on_the_cache_dtype():
    rng = np.random.Generator(np.random.PCG64(4))
    k = rng.standard_normal((5, 2, 16)).astype(np.float32)
    v = rng.standard_normal((5, 2, 16)).astype(np.float32)
    slots = np.array([3, 17, 40, 2, 63])
    for dt, quant in ((np.int8, int8_quantize_rows), (np.uint8, fp8_quantize_rows)):
        kc = np.zeros((4, 2, 16, 16), dt)
        vc = np.zeros_like(kc)
        ks = np.zeros((4, 16), np.float32)
        vs = np.zeros_like(ks)
        kc, vc, ks, vs = cache_write(k, v, slots, kc, vc, ks, vs)
        kq, kscale = quant(k)
        assert np.array_equal(kc[slots // 16, :, slots % 16, :], kq)
        assert np.array_equal(ks[slots // 16, slots % 16], kscale)


def test_attention_over_int8_equals_attention_over_the_same_values_as_floats():
    rng = np.random.Generator(np.random.PCG64(5))
    nb, H, D = 6, 2, 16
    kf = rng.standard_normal((nb * 16, H, D)).astype(np.float32)
    vf = rng.standard_normal((nb * 16, H, D)).astype(np.float32)
    kc8, ks = int8_quantize_rows(kf)
    vc8, vs = int8_quantize_rows(vf)
    to_cache = lambda a: a.reshape(nb, 16, H, D).transpose(0, 2, 1, 3).copy()
    kc, vc = to_cache(kc8), to_cache(vc8)
    kdeq = to_cache(kc8.astype(np.float64) * ks[:, None, None])
    vdeq = to_cache(vc8.astype(np.float64) * vs[:, None, None])
    tables = rng.permutation(nb)[None, :].repeat(2, 0)
    lens = np.array([77, 96])
    q = rng.standard_normal((2, 4, D))
    a = paged_decode(q, kc, vc, tables, lens, 0.3, ks.reshape(nb, 16), vs.reshape(nb, 16))
    b = paged_decode(q, kdeq, vdeq, tables, lens, 0.3)
    assert np.array_equal(a, b)
