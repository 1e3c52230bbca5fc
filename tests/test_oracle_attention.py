"""Pins for the oracle's paged decode attention.

The pages print no worked attention example, so the oracle is pinned to what
the mathematics fixes: a de-paged brute force through an independent library
routine (torch scaled_dot_product_attention in float64), invariance under a
relabelling of physical blocks, closed forms (one-token context, equal keys,
zero query, constant values), grouped-query equivalence to multi-head
attention with repeated K/V heads, and softmax rows summing to one.
"""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode, softmax_weights, gather_kv
from oracle.cache_ops import fp8_quantize_token
from oracle.fp8_e4m3 import e4m3_decode

BS = 16


def _contiguous_case(seed, B, Hq, Hkv, D, lens, spare=5):
    """Contiguous per-sequence K/V, then paged into a shuffled pool by the test."""
    rng = np.random.Generator(np.random.PCG64(seed))
    nblk = [-(-n // BS) for n in lens]
    pool = sum(nblk) + spare
    perm = rng.permutation(pool)
    maxb = max(max(nblk), 1)
    tables = np.full((B, maxb), -1, np.int64)
    kc = rng.standard_normal((pool, Hkv, BS, D))
    vc = rng.standard_normal((pool, Hkv, BS, D))
    Ks, Vs = [], []
    pos = 0
    for b, n in enumerate(lens):
        Kseq = rng.standard_normal((n, Hkv, D))
        Vseq = rng.standard_normal((n, Hkv, D))
        tables[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
        for t in range(n):                       # page the contiguous rows
            kc[tables[b, t // BS], :, t % BS, :] = Kseq[t]
            vc[tables[b, t // BS], :, t % BS, :] = Vseq[t]
        Ks.append(Kseq)
        Vs.append(Vseq)
    q = rng.standard_normal((B, Hq, D))
    return q, kc, vc, tables, np.array(lens), Ks, Vs


def _sdpa(q_bh, Kseq, Vseq, G, scale):
    """torch SDPA in float64 on contiguous K/V, GQA by repeating kv heads."""
    qt = torch.from_numpy(q_bh)[:, None, :]                         # [Hq, 1, D]
    kt = torch.from_numpy(Kseq).permute(1, 0, 2).repeat_interleave(G, 0)  # [Hq, n, D]
    vt = torch.from_numpy(Vseq).permute(1, 0, 2).repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[:, 0, :].numpy()


@pytest.mark.parametrize("Hq,Hkv,D,lens", [
    (4, 4, 64, [5, 17, 32, 47]),
    (8, 2, 32, [1, 16, 33, 100, 15]),
    (8, 1, 16, [64, 3]),
])
def test_matches_depaged_sdpa(Hq, Hkv, D, lens):
    scale = 1 / np.sqrt(D)
    q, kc, vc, tab, L, Ks, Vs = _contiguous_case(11, len(lens), Hq, Hkv, D, lens)
    out = paged_decode(q, kc, vc, tab, L, scale)
    for b in range(len(lens)):
        ref = _sdpa(q[b], Ks[b], Vs[b], Hq // Hkv, scale)
        np.testing.assert_allclose(out[b], ref, atol=1e-12, rtol=1e-12)


def test_physical_block_relabelling_is_invisible():
    q, kc, vc, tab, L, _, _ = _contiguous_case(12, 3, 4, 2, 32, [40, 7, 16])
    rng = np.random.Generator(np.random.PCG64(3))
    pi = rng.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    tab2 = np.where(tab >= 0, pi[np.maximum(tab, 0)], -1)
    a = paged_decode(q, kc, vc, tab, L, 0.3)
    b = paged_decode(q, kc2, vc2, tab2, L, 0.3)
    assert np.array_equal(a, b)


def test_closed_forms():
    q, kc, vc, tab, L, Ks, Vs = _contiguous_case(13, 2, 2, 2, 16, [1, 30])
    out = paged_decode(q, kc, vc, tab, L, 0.25)
    assert np.array_equal(out[0], Vs[0][0])          # one token: out = V_0 exactly
    # equal keys or a zero query -> uniform weights -> mean of V
    kc_eq = kc.copy()
    kc_eq[:] = kc[tab[1, 0], :, 0, :][None, :, None, :]
    mean = Vs[1].mean(axis=0)
    np.testing.assert_allclose(paged_decode(q, kc_eq, vc, tab, L, 0.25)[1], mean, atol=1e-13)
    np.testing.assert_allclose(paged_decode(np.zeros_like(q), kc, vc, tab, L, 0.25)[1], mean, atol=1e-13)
    # constant V -> constant output
    out1 = paged_decode(q, kc, np.full_like(vc, 1.5), tab, L, 0.25)
    np.testing.assert_allclose(out1, 1.5, atol=1e-13)
    # empty context -> zeros
    assert not paged_decode(q, kc, vc, tab, np.array([0, 0]), 0.25).any()


def test_grouped_query_equals_repeated_mha():
    q, kc, vc, tab, L, _, _ = _contiguous_case(14, 2, 8, 2, 16, [21, 50])
    gqa = paged_decode(q, kc, vc, tab, L, 0.2)
    mha = paged_decode(q, np.repeat(kc, 4, axis=1), np.repeat(vc, 4, axis=1), tab, L, 0.2)
    assert np.array_equal(gqa, mha)


def test_softmax_rows_sum_to_one():
    rng = np.random.Generator(np.random.PCG64(5))
    for n in (1, 2, 17, 300):
        K = rng.standard_normal((n, 24)) * 4
        p = softmax_weights(rng.standard_normal(24), K, 0.7)
        assert p.min() >= 0 and abs(p.sum() - 1) < 1e-14


def test_fp8_cache_is_decoded_with_its_scales():
    q, kc, vc, tab, L, Ks, Vs = _contiguous_case(15, 2, 4, 2, 32, [19, 33])
    kq = np.zeros(kc.shape, np.uint8)
    vq = np.zeros(vc.shape, np.uint8)
    ks = np.ones(kc.shape[0:1] + (BS,), np.float32)
    vs = np.ones_like(ks)
    for blk in range(kc.shape[0]):
        for r in range(BS):
            kq[blk, :, r, :], ks[blk, r] = fp8_quantize_token(kc[blk, :, r, :].astype(np.float32))
            vq[blk, :, r, :], vs[blk, r] = fp8_quantize_token(vc[blk, :, r, :].astype(np.float32))
    out = paged_decode(q, kq, vq, tab, L, 0.2, ks, vs)
    for b in range(2):
        Kd = np.stack([e4m3_decode(kq[tab[b, t // BS], :, t % BS, :]) * ks[tab[b, t // BS], t % BS]
                       for t in range(L[b])])
        Vd = np.stack([e4m3_decode(vq[tab[b, t // BS], :, t % BS, :]) * vs[tab[b, t // BS], t % BS]
                       for t in range(L[b])])
        np.testing.assert_allclose(out[b], _sdpa(q[b], Kd, Vd, 2, 0.2), atol=1e-12)
    # and the dequantised cache is close to the unquantised one
    np.testing.assert_allclose(out, paged_decode(q, kc, vc, tab, L, 0.2), atol=0.1)


def test_gather_reads_through_the_table():
    q, kc, vc, tab, L, Ks, Vs = _contiguous_case(16, 1, 2, 2, 8, [37])
    for g in range(2):
        assert np.array_equal(gather_kv(kc, tab[0], 37, g), Ks[0][:, g, :])
        assert np.array_equal(gather_kv(vc, tab[0], 37, g), Vs[0][:, g, :])
