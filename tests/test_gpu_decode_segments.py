"""pa_decode_append_segments (each block shared by any subset of a group's
members read once) against the oracle and against the plain
pa_decode_append.

Groups are built as beam search leaves them after reselection: every member
shares the prompt's blocks, pairs of members share a parent's further blocks,
and each member has a private tail holding its last token.  The items come
from ops.shared_table_segments.  Outputs must match the oracle within the
attention tolerance and the plain call within 5e-4 (the partitions differ);
the fused writes must leave the same caches.  Shapes cover G = 1, 2, 4, 8,
16-bit and 1-byte caches, items cut to 3 blocks, an empty member, a call with
no items, and the flags for bad items and members whose blocks differ."""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode
from oracle.cache_ops import cache_write as o_write
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, assert_close, requires_cuda
from tests.test_gpu_decode_grouped import caches, last_slots

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


def tree_case(seed, Hq, Hkv, kv, D=128, groups=3, size=4, prompt=5, zero=()):
    """Member lengths 16 * (prompt + pair + own) - r; members share the
    prompt's blocks, each pair (2i, 2i+1) shares `pair` more, the rest is
    private (the last block always is)."""
    rng = W.rng_for(seed)
    lens, share = [], []
    for _ in range(groups):
        pairs = [int(rng.integers(0, 4)) for _ in range((size + 1) // 2)]
        for m in range(size):
            own = int(rng.integers(1, 4))
            lens.append(16 * (prompt + pairs[m // 2] + own) - int(rng.integers(0, 16)))
            share.append(pairs[m // 2])
    for b in zero:
        lens[b] = 0
    w = W.make_decode(f"tree{seed}", seed + 5, len(lens), Hq, Hkv, D, kv, lens, pool_factor=1.3)
    start = np.arange(0, groups * size + 1, size, dtype=np.int32)
    t = w.block_tables.copy()
    for k in range(groups):
        g0 = start[k]
        for m in range(1, size):
            b = g0 + m
            if lens[b] == 0 or lens[g0] == 0:
                continue
            t[b, :prompt] = t[g0, :prompt]
            if m % 2 == 1 and lens[b - 1] > 0:
                t[b, prompt:prompt + share[b]] = t[b - 1, prompt:prompt + share[b]]
    w.block_tables = t
    return w, start


def run(w, start, bpi=32, plain=False, items=None, max_items=None):
    rng = W.rng_for(17)
    q = w.q.to(torch.bfloat16) if w.kv_dtype == "bf16" else w.q
    k_new = W.randn(rng, (w.B, w.Hkv, w.D), q.dtype).to(DEV)
    v_new = W.randn(rng, (w.B, w.Hkv, w.D), q.dtype).to(DEV)
    sl = torch.from_numpy(last_slots(w)).to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables, dtype=np.int32)).to(DEV)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens, dtype=np.int32)).to(DEV)
    ml = max(int(w.context_lens.max()), 1)
    kc, vc, ks, vs = caches(w)
    if plain:
        out = ops.decode_append(k_new, v_new, sl, q.to(DEV), kc, vc, bt, cl, ml, w.scale, out_dtype=torch.float32,
                                k_scale=ks, v_scale=vs)
    else:
        most = None
        if items is None:
            items, most = ops.shared_table_segments(w.block_tables, w.context_lens, start, bpi)
        mi = max_items or max(most or 0, 1)
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
        ops.decode_append_segments(k_new, v_new, sl, q.to(DEV), kc, vc, bt, cl, ml, w.scale,
                                   torch.from_numpy(start).to(DEV), torch.from_numpy(items).to(DEV).view(-1, 4),
                                   int(np.diff(start).max()), mi, out=out, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out.cpu().numpy(), [t.cpu() if t is not None else None for t in (kc, vc, ks, vs)], (k_new, v_new, q)


CASES = [  # Hq, Hkv, kv, group size, items of at most bpi blocks
    (8, 8, "f16", 4, 32),
    (16, 8, "f16", 4, 3),
    (16, 8, "bf16", 4, 32),
    (8, 2, "f16", 2, 2),
    (32, 4, "bf16", 1, 32),
    (8, 8, "fp8", 4, 3),
    (16, 8, "int8", 4, 32),
    (4, 4, "bf16", 8, 5),
]


@pytest.mark.parametrize("Hq,Hkv,kv,size,bpi", CASES, ids=lambda v: str(v))
def test_segments_match_oracle_and_plain(Hq, Hkv, kv, size, bpi):
    D = 64 if (Hq, Hkv) == (4, 4) else 128
    w, start = tree_case(70 + Hq + Hkv + size, Hq, Hkv, kv, D=D, size=size)
    items, _ = ops.shared_table_segments(w.block_tables, w.context_lens, start, bpi)
    if size > 1:  # the tree is exercised: items shared by the whole group and by pairs
        nms = (items[:, 3] >> 8) & 0xff
        assert (nms == size).any() and ((nms > 1) & (nms < size)).any() or size == 2
    got, dev_caches, (k_new, v_new, q) = run(w, start, bpi)
    plain, plain_caches, _ = run(w, start, plain=True)
    for a, b in zip(dev_caches, plain_caches):
        assert a is None or torch.equal(a, b)
    assert np.abs(got - plain).max() <= 5e-4, float(np.abs(got - plain).max())
    if kv in ("fp8", "int8"):
        kc, vc, ks, vs = (t.numpy() for t in dev_caches)
        ref = paged_decode(np_exact(q), kc, vc, w.block_tables, w.context_lens, w.scale, k_scale=ks, v_scale=vs)
    else:
        okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), last_slots(w), np_exact(w.k_pool),
                                 np_exact(w.v_pool))
        assert np.array_equal(np_exact(dev_caches[0]), okc) and np.array_equal(np_exact(dev_caches[1]), ovc)
        ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL[kv], f"segments {Hq}/{Hkv} {kv} size {size} bpi {bpi}")


def test_members_in_more_than_32_items():
    """One-block items over a 40-block prompt: every member is listed by more
    than 32 items, which the merge takes chunk by chunk."""
    w, start = tree_case(85, 8, 8, "f16", prompt=40)
    items, _ = ops.shared_table_segments(w.block_tables, w.context_lens, start, 1)
    got, _, (k_new, v_new, q) = run(w, start, bpi=1)
    okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), last_slots(w), np_exact(w.k_pool),
                             np_exact(w.v_pool))
    ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL["f16"], "one-block items")


def test_empty_member_and_no_items():
    """An empty member is in no item and gets zero rows; with no items at all
    every row is zero."""
    w, start = tree_case(81, 8, 8, "f16", zero=(5,))
    got, _, (k_new, v_new, q) = run(w, start)
    assert np.all(got[5] == 0.0)
    okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), last_slots(w), np_exact(w.k_pool),
                             np_exact(w.v_pool))
    assert_close(got, paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale), TOL["f16"],
                 "empty member")
    none = np.zeros((0, 4), np.int32)
    got, _, _ = run(w, start, items=none, max_items=4)
    assert np.all(got == 0.0)


def test_bad_items_and_differing_blocks_are_flagged():
    w, start = tree_case(83, 8, 8, "f16")
    items, most = ops.shared_table_segments(w.block_tables, w.context_lens, start, 32)
    bad = items.copy()
    k = int(np.argmax((bad[:, 3] >> 8) & 0xff))
    bad[k, 1] = (bad[k, 1] & ~0xf) | 9  # member 9 of a group of 4
    run(w, start, items=bad, max_items=most)
    assert ops.device_errors(clear=True) & ops.DEVERR_GROUP
    bad = items.copy()
    bad[0, 3] = (bad[0, 3] & 0xffff) | (most << 16)  # a slot past the bound
    run(w, start, items=bad, max_items=most)
    assert ops.device_errors(clear=True) & ops.DEVERR_GROUP
    w.block_tables[1, 0] = w.block_tables[1, w.context_lens[1] // 16 - 1]  # member 1 leaves the prompt's block 0
    run(w, start, items=items, max_items=most)
    assert ops.device_errors(clear=True) & ops.DEVERR_GROUP


@pytest.mark.parametrize("cfg", ["gqa70b_b64", "llama7b_b32"])
def test_one_member_groups_full_size_all_rows(cfg):
    """A batch without sharing as B one-member groups: the items are each
    sequence's live partitions, cut with the partition length
    pa_decode_items_plan gives.  At the full workload size every row matches
    the oracle, the plain call within 5e-4, and the fused writes leave the
    same caches.  The log-uniform GQA batch is one the planner lists; the
    uniform llama batch is one it leaves on the fixed grid (run here anyway)."""
    w = W.CONFIGS[cfg]()
    start = np.arange(w.B + 1, dtype=np.int32)
    ml = int(w.context_lens.max())
    kc_probe = torch.empty((1, w.Hkv, 16, w.D), dtype=w.q.dtype)
    use, bpi, most = ops.decode_items_plan(w.context_lens, w.Hq, ml, kc_probe)
    assert use == (cfg == "gqa70b_b64")
    items, slots = ops.shared_table_segments(w.block_tables, w.context_lens, start, bpi)
    assert slots <= most and ((items[:, 3] >> 8) & 0xff == 1).all()
    got, dev_caches, (k_new, v_new, q) = run(w, start, bpi, items=items, max_items=most)
    plain, plain_caches, _ = run(w, start, plain=True)
    for a, b in zip(dev_caches, plain_caches):
        assert a is None or torch.equal(a, b)
    assert np.abs(got - plain).max() <= 5e-4, float(np.abs(got - plain).max())
    okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), last_slots(w), np_exact(w.k_pool),
                             np_exact(w.v_pool))
    ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL[w.kv_dtype], f"{cfg} one-member groups")


@pytest.mark.parametrize("kv", ["f16", "fp8"])
@pytest.mark.parametrize("bpi", [4, 1])
def test_one_member_groups_edge_lengths(kv, bpi):
    """One-member groups over lengths 0, 5, 16, 17, 300 and 1100, items of 4
    blocks (at most 18 a member) and of one block (69 for the longest: the
    merge takes them in three chunks).  An empty member gets zero rows and
    every row matches the oracle and the plain call; a second launch on the
    same inputs gives the same rows."""
    lens = [0, 5, 16, 17, 300, 1100]
    w = W.make_decode(f"edges{bpi}{kv}", 61, len(lens), 8, 4, 128, kv, lens, pool_factor=1.2)
    start = np.arange(w.B + 1, dtype=np.int32)
    items, most = ops.shared_table_segments(w.block_tables, w.context_lens, start, bpi)
    assert most == -(-69 // bpi)
    got, dev_caches, (k_new, v_new, q) = run(w, start, bpi, items=items, max_items=most)
    assert np.all(got[0] == 0.0)
    plain, plain_caches, _ = run(w, start, plain=True)
    for a, b in zip(dev_caches, plain_caches):
        assert a is None or torch.equal(a, b)
    assert np.abs(got - plain).max() <= 5e-4, float(np.abs(got - plain).max())
    if kv == "fp8":
        kc, vc, ks, vs = (t.numpy() for t in dev_caches)
        ref = paged_decode(np_exact(q), kc, vc, w.block_tables, w.context_lens, w.scale, k_scale=ks, v_scale=vs)
    else:
        okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), last_slots(w), np_exact(w.k_pool),
                                 np_exact(w.v_pool))
        ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL[kv], f"one-member edges {kv} bpi {bpi}")
    again, _, _ = run(w, start, bpi, items=items, max_items=most)
    assert np.array_equal(again, got)
