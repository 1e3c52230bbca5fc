"""Pins for the oracle's multi-token paged attention (chunked prefill and
speculative verification).

Nothing on the pages prints a worked example, so the oracle is pinned to
what the mathematics fixes, each check able to catch a different plausible
mistake:

* a chunk's rows equal the last n rows of one causal pass over the whole
  sequence, computed by torch scaled_dot_product_attention(is_causal=True)
  in float64 on de-paged K/V (an off-by-one in the chunk offset, a wrong
  mask direction, a wrong kv-head mapping or a transposed operand fails);
* with all keys equal the weights are uniform, so row i is the mean of
  V[0 .. L-n+i] (the exact causal boundary, in closed form);
* one query token per sequence reduces to paged decode;
* a perturbation of the key/value at position pos+1 leaves row pos alone
  and changes the row after it (causality, both directions);
* relabelling physical blocks changes nothing (paging is transparent);
* a prompt run as two chunks gives the rows of one chunk (chunking).
"""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode, paged_prefill

BS = 16


def _case(seed, Hq, Hkv, D, lens, nq, spare=3):
    """Contiguous per-sequence K/V paged into a shuffled pool, plus packed queries."""
    rng = np.random.Generator(np.random.PCG64(seed))
    nblk = [-(-n // BS) for n in lens]
    pool = sum(nblk) + spare
    perm = rng.permutation(pool)
    tables = np.full((len(lens), max(max(nblk), 1)), -1, np.int64)
    kc = rng.standard_normal((pool, Hkv, BS, D))
    vc = rng.standard_normal((pool, Hkv, BS, D))
    Ks, Vs = [], []
    pos = 0
    for b, n in enumerate(lens):
        Kseq = rng.standard_normal((n, Hkv, D))
        Vseq = rng.standard_normal((n, Hkv, D))
        tables[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
        for t in range(n):
            kc[tables[b, t // BS], :, t % BS, :] = Kseq[t]
            vc[tables[b, t // BS], :, t % BS, :] = Vseq[t]
        Ks.append(Kseq)
        Vs.append(Vseq)
    q_start = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    q = rng.standard_normal((int(q_start[-1]), Hq, D))
    return q, q_start, kc, vc, tables, np.array(lens), Ks, Vs


def _sdpa_causal_tail(q_rows, Kseq, Vseq, G, scale):
    """Last n rows of a full causal pass: the chunk's queries are placed at
    the last n positions of a length-L query sequence whose other rows are
    zeros (they do not influence the last rows under a causal mask)."""
    n = q_rows.shape[0]
    L = Kseq.shape[0]
    Hq = q_rows.shape[1]
    qfull = torch.zeros((Hq, L, q_rows.shape[2]), dtype=torch.float64)
    qfull[:, L - n:, :] = torch.from_numpy(q_rows).permute(1, 0, 2)
    kt = torch.from_numpy(Kseq).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(Vseq).permute(1, 0, 2).repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qfull, kt, vt, is_causal=True, scale=scale)
    return o[:, L - n:, :].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv,D,lens,nq", [
    (4, 4, 32, [5, 17, 40, 33], [5, 3, 40, 1]),
    (8, 2, 16, [64, 100, 16, 1], [17, 64, 16, 1]),
    (6, 1, 8, [31, 48], [31, 7]),
])
def test_chunk_equals_tail_of_full_causal_pass(Hq, Hkv, D, lens, nq):
    q, qs, kc, vc, tab, L, Ks, Vs = _case(3, Hq, Hkv, D, lens, nq)
    scale = 0.37
    got = paged_prefill(q, qs, kc, vc, tab, L, scale)
    for b in range(len(lens)):
        want = _sdpa_causal_tail(q[qs[b]:qs[b + 1]], Ks[b], Vs[b], Hq // Hkv, scale)
        assert np.abs(got[qs[b]:qs[b + 1]] - want).max() < 1e-12, f"sequence {b}"


def test_equal_keys_give_running_means_of_values():
    Hq, Hkv, D, lens, nq = 2, 1, 8, [37, 20], [37, 9]
    q, qs, kc, vc, tab, L, Ks, Vs = _case(4, Hq, Hkv, D, lens, nq)
    kc[:] = 0.25  # every key identical -> every score identical
    got = paged_prefill(q, qs, kc, vc, tab, L, 1.0)
    for b in range(2):
        n = nq[b]
        for i in range(n):
            pos = lens[b] - n + i
            want = Vs[b][:pos + 1, 0, :].mean(axis=0)
            for h in range(Hq):
                assert np.abs(got[qs[b] + i, h] - want).max() < 1e-13


def test_single_token_queries_reduce_to_decode():
    Hq, Hkv, D, lens = 8, 2, 16, [1, 15, 16, 17, 90]
    q, qs, kc, vc, tab, L, _, _ = _case(5, Hq, Hkv, D, lens, [1] * 5)
    got = paged_prefill(q, qs, kc, vc, tab, L, 0.5)
    want = paged_decode(q, kc, vc, tab, L, 0.5)
    assert np.abs(got - want).max() < 1e-13


def test_causality_both_directions():
    Hq, Hkv, D, lens, nq = 2, 2, 8, [40], [12]
    q, qs, kc, vc, tab, L, _, _ = _case(6, Hq, Hkv, D, lens, nq)
    base = paged_prefill(q, qs, kc, vc, tab, L, 1.0)
    i = 5
    pos = lens[0] - nq[0] + i
    nxt = pos + 1
    for cache in ("k", "v"):
        k2, v2 = kc.copy(), vc.copy()
        tgt = k2 if cache == "k" else v2
        tgt[tab[0, nxt // BS], :, nxt % BS, :] += 3.0
        o = paged_prefill(q, qs, k2, v2, tab, L, 1.0)
        assert np.array_equal(o[:i + 1], base[:i + 1]), "a row saw a later key"
        assert np.abs(o[i + 1] - base[i + 1]).max() > 1e-6, "a row missed its own key"


def test_block_relabelling_is_transparent():
    Hq, Hkv, D, lens, nq = 4, 2, 8, [50, 23], [20, 23]
    q, qs, kc, vc, tab, L, _, _ = _case(7, Hq, Hkv, D, lens, nq, spare=6)
    base = paged_prefill(q, qs, kc, vc, tab, L, 0.7)
    rng = np.random.Generator(np.random.PCG64(1))
    perm = rng.permutation(kc.shape[0])            # new id of old block b = perm[b]
    k2, v2 = np.empty_like(kc), np.empty_like(vc)
    k2[perm], v2[perm] = kc, vc
    tab2 = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1)
    assert np.array_equal(paged_prefill(q, qs, k2, v2, tab2, L, 0.7), base)


def test_two_chunks_equal_one_chunk():
    Hq, Hkv, D, lens = 4, 4, 16, [70]
    q, qs, kc, vc, tab, L, _, _ = _case(8, Hq, Hkv, D, lens, [70])
    whole = paged_prefill(q, qs, kc, vc, tab, L, 0.3)
    a = 29  # first chunk: tokens [0, a) with context a; second: [a, 70) with context 70
    first = paged_prefill(q[:a], [0, a], kc, vc, tab, [a], 0.3)
    second = paged_prefill(q[a:], [0, 70 - a], kc, vc, tab, [70], 0.3)
    assert np.array_equal(np.concatenate([first, second]), whole)


def test_empty_sequences_and_invalid_tokens():
    Hq, Hkv, D, lens, nq = 2, 1, 8, [0, 10, 3], [0, 4, 5]
    q, qs, kc, vc, tab, L, _, _ = _case(9, Hq, Hkv, D, [max(n, 1) for n in lens], nq)
    got = paged_prefill(q, qs, kc, vc, tab, np.array(lens), 1.0)
    # sequence 2 has 5 queries but 3 keys: its first two tokens have none
    assert np.array_equal(got[4:6], np.zeros((2, Hq, D)))
    assert np.abs(got[6:9]).max() > 0
