"""Pins for the oracle's E4M3 codec against the format definition and torch.

The oracle codec is written from the OCP E4M3 definition; these tests tie it
to (a) the specification's own code/value table (golden fixture), (b) an
independent library implementation (torch.float8_e4m3fn casts) over every
code and over a million float32 values, and (c) the round-to-nearest-even and
saturation rules at every midpoint of the grid.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle.fp8_e4m3 import e4m3_decode, e4m3_encode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spec_values.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        rows.append((int(code, 16), float(val)))
    return rows


def test_decode_matches_spec_table():
    for code, val in _golden():
        got = e4m3_decode(np.array([code], np.uint8))[0]
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_encode_roundtrips_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_decode(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(e4m3_encode(vals[finite]), codes[finite])


def test_encode_ties_go_to_even_code():
    pos = np.arange(0, 0x7E, dtype=np.uint8)          # 0 .. 416 (next is 448)
    lo, hi = e4m3_decode(pos), e4m3_decode(pos + 1)
    mid = (lo + hi) / 2                                 # exact in float64
    got = e4m3_encode(mid)
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    # just off the midpoint rounds to the nearer neighbour
    eps = (hi - lo) * 1e-3
    assert np.array_equal(e4m3_encode(mid - eps), pos)
    assert np.array_equal(e4m3_encode(mid + eps), (pos + 1).astype(np.uint8))
    assert np.array_equal(e4m3_encode(-mid), want | 0x80)


def test_encode_saturates_and_keeps_signed_zero():
    assert e4m3_encode(np.array([448.0, 449.0, 1e6, np.inf]))[:].tolist() == [0x7E] * 4
    assert e4m3_encode(np.array([-448.0, -1e30, -np.inf])).tolist() == [0xFE] * 3
    assert e4m3_encode(np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11)])).tolist() == [0, 0x80, 0, 0x80]
    assert e4m3_encode(np.array([np.nan])).tolist() == [0x7F]


def test_encode_matches_torch_on_a_million_floats():
    rng = np.random.Generator(np.random.PCG64(7))
    mag = np.exp(rng.uniform(math.log(2.0 ** -12), math.log(460.0), size=1_000_000))
    x = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode(x)
    assert np.array_equal(got, ref)
