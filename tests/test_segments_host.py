"""ops.shared_table_segments: the host helper that lists, per group, the runs
of table positions a subset of the members all hold (no GPU).  Checked
against its definition written out position by position, and against the
property the segment decode relies on: every block a member holds is in
exactly one item listing it, and a physical block shared by several members
is read once."""
import numpy as np
import pytest

from paged_kv_cache_191_gb300 import ops
from tests.libfixture import palib  # noqa: F401


def segments_by_definition(tables, lens, gs, bpi):
    """Position by position: the class of member m at position j is the set
    of members holding the same block there, unless j is not before every
    such member's last block (then m alone); a segment is a maximal run of
    positions with the same class, cut into pieces of bpi blocks."""
    out = []
    for k in range(len(gs) - 1):
        members = list(range(gs[k], gs[k + 1]))
        nblk = {b: -(-int(lens[b]) // 16) for b in members}
        last = {b: (int(lens[b]) - 1) // 16 if lens[b] > 0 else -1 for b in members}

        def cls(b, j):
            same = [c for c in members if j < nblk[c] and tables[c][j] == tables[b][j] and j < last[c]]
            return tuple(same) if b in same and len(same) > 1 else (b,)

        for b in members:
            j = 0
            while j < nblk[b]:
                c = cls(b, j)
                j1 = j + 1
                while j1 < nblk[b] and cls(b, j1) == c:
                    j1 += 1
                if c[0] == b:  # the class's first member lists it
                    for p0 in range(j, j1, bpi):
                        out.append((k, tuple(m - gs[k] for m in c), p0, min(bpi, j1 - p0)))
                j = j1
    return sorted(out)


def decode_items(items):
    """(group, members, first block, blocks) of each item, sorted."""
    res = []
    for k, ml, j0, w in items.tolist():
        nm = (w >> 8) & 0xff
        res.append((k, tuple(((ml & 0xffffffff) >> (4 * i)) & 15 for i in range(nm)), j0, w & 0xff))
    return sorted(res)


def slots_of(items):
    return [((w & 0xffffffff) >> 16) & 0xffff for w in items[:, 3].tolist()]


def tree_tables(rng, n_groups, size, prompt_blocks, max_tail):
    """Beam-like groups: all members share the prompt's blocks, then pairs of
    members share a few more (a parent's blocks after reselection), then
    private tails.  Block ids are drawn without reuse across groups."""
    ids = iter(rng.permutation(100000))
    rows, lens = [], []
    for _ in range(n_groups):
        base = [next(ids) for _ in range(prompt_blocks)]
        pair_extra = {}
        for m in range(size):
            pair = m // 2
            if pair not in pair_extra:
                pair_extra[pair] = [next(ids) for _ in range(int(rng.integers(0, 4)))]
            own = [next(ids) for _ in range(int(rng.integers(1, max_tail + 1)))]
            row = base + pair_extra[pair] + own
            rows.append(row)
            lens.append(16 * (len(row) - 1) + int(rng.integers(1, 17)))
    width = max(len(r) for r in rows)
    tables = np.full((len(rows), width), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = r
    gs = np.arange(0, n_groups * size + 1, size, dtype=np.int32)
    return tables, np.array(lens, np.int32), gs


@pytest.mark.parametrize("seed,size,bpi", [(1, 4, 32), (2, 4, 3), (3, 2, 1), (4, 8, 7), (5, 1, 64)])
def test_segments_match_their_definition(seed, size, bpi):
    rng = np.random.default_rng(seed)
    tables, lens, gs = tree_tables(rng, 5, size, int(rng.integers(0, 9)), 5)
    items, most = ops.shared_table_segments(tables, lens, gs, bpi)
    assert decode_items(items) == segments_by_definition(tables, lens, gs, bpi)
    # longest first; a group's items hold slots 0 .. n_k - 1, in (owner, position) order
    nb = items[:, 3] & 0xff
    assert (np.diff(nb) <= 0).all()
    slots = slots_of(items)
    for k in range(len(gs) - 1):
        mine = [i for i in range(len(items)) if items[i, 0] == k]
        assert sorted(slots[i] for i in mine) == list(range(len(mine)))
        by_slot = sorted(mine, key=lambda i: slots[i])
        firsts = [(int(items[i, 1]) & 15, int(items[i, 2])) for i in by_slot]
        assert firsts == sorted(firsts)
    assert most == max(np.bincount(items[:, 0], minlength=len(gs) - 1))


def test_every_block_is_read_once():
    """Coverage: each (member, position) below its block count is in exactly
    one item listing it; the listed members hold the same block there; a
    multi-member item lies before each member's last block; and the items'
    blocks add up to the group's distinct (position, block) pairs."""
    rng = np.random.default_rng(9)
    tables, lens, gs = tree_tables(rng, 6, 4, 12, 6)
    lens[3] = 0  # an empty member holds nothing
    items, _ = ops.shared_table_segments(tables, lens, gs, 8)
    seen = {}
    for k, ml, j0, nb, members in ((k, ml, j0, nb, m) for k, ml, j0, nb_w in items.tolist()
                                   for nb, m in [(nb_w & 0xff, [((ml & 0xffffffff) >> (4 * i)) & 15
                                                                for i in range((nb_w >> 8) & 0xff)])]):
        assert members == sorted(members) and len(set(members)) == len(members)
        seqs = [gs[k] + m for m in members]
        for j in range(j0, j0 + nb):
            ids = {int(tables[b][j]) for b in seqs}
            assert len(ids) == 1
            for b in seqs:
                assert j < -(-int(lens[b]) // 16)
                if len(seqs) > 1:
                    assert j < (int(lens[b]) - 1) // 16
                assert (b, j) not in seen
                seen[(b, j)] = True
    for b in range(len(lens)):
        for j in range(-(-int(lens[b]) // 16)):
            assert (b, j) in seen
    for k in range(len(gs) - 1):
        distinct = {(j, int(tables[b][j])) for b in range(gs[k], gs[k + 1]) for j in range(-(-int(lens[b]) // 16))}
        nb = sum(w & 0xff for kk, _, _, w in items.tolist() if kk == k)
        # the last blocks are private here, so every distinct block is one item position
        assert nb == len(distinct)


def test_shared_last_block_is_read_per_member():
    """Two members claiming the same block at their last position (a missed
    copy on write) read it separately: the fused write lands there."""
    tables = np.array([[7, 8], [7, 8]], np.int32)
    items, _ = ops.shared_table_segments(tables, np.array([20, 25]), np.array([0, 2]), 32)
    assert decode_items(items) == [(0, (0,), 1, 1), (0, (0, 1), 0, 1), (0, (1,), 1, 1)]


def test_bad_arguments():
    with pytest.raises(ValueError):
        ops.shared_table_segments(np.zeros((9, 2), np.int32), np.ones(9), np.array([0, 9]), 32)
    with pytest.raises(ValueError):
        ops.shared_table_segments(np.zeros((2, 2), np.int32), np.ones(2), np.array([0, 2]), 65)


def test_workspace_size(palib):
    d = ops.CacheDesc(num_blocks=8, num_kv_heads=2, head_dim=128, block_size=16, kv_dtype=ops.F16)
    import ctypes as C
    ws = palib.pa_decode_segments_workspace_size(6, 4, 2, 4, 10, C.byref(d))
    assert ws == (6 * 4 * 10 * (128 + 2) * 4 + 255) // 256 * 256
    assert palib.pa_decode_segments_workspace_size(6, 4, 2, 4, 0, C.byref(d)) == 0
    assert palib.pa_decode_segments_workspace_size(6, 4, 2, 9, 10, C.byref(d)) == 0
