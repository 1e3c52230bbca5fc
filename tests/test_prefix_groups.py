"""ops.prefix_groups: the host helper that finds shared-prefix groups for the
grouped decode (no GPU)."""
import numpy as np
import pytest

from paged_kv_cache_191_gb300 import ops
from tests.libfixture import palib  # noqa: F401


def test_forked_beams_form_groups_with_their_prompt_prefix(palib):
    """Beams forked from two prompts (64 + 3 blocks) and grown by private
    tails: one group per prompt, prefix = the prompt's whole blocks."""
    a = ops.BlockAllocator(200)
    a.alloc_seq(1000, 64 * 16)        # prompt 1: 64 full blocks
    a.alloc_seq(1001, 3 * 16 + 5)     # prompt 2: 3 full blocks and 5 tokens
    beams = list(range(7))
    a.fork_seqs([1000] * 4 + [1001] * 3, beams)
    for i, t in enumerate([1, 20, 33, 7, 11, 2, 40]):
        a.append_tokens(i, t, want_slots=False)
    tables, lens = a.tables(beams, 80)
    gs, pre = ops.prefix_groups(tables, lens, 4)
    assert gs.tolist() == [0, 4, 7]
    # prompt 2's partial block is copied on write by the first append to it, so
    # only its 3 full blocks stay shared
    assert pre.tolist() == [64, 3]


@pytest.mark.parametrize("max_size", [1, 2, 3])
def test_group_size_bound_and_singletons(max_size):
    tables = np.array([[5, 6, 7, 8], [5, 6, 9, 10], [5, 6, 7, 11], [20, 21, 22, 23]])
    lens = np.array([64, 64, 64, 64])  # 4 blocks each; 3 usable before the last token
    gs, pre = ops.prefix_groups(tables, lens, max_size)
    want = {1: ([0, 1, 2, 3, 4], [0, 0, 0, 0]), 2: ([0, 2, 3, 4], [2, 0, 0]),
            3: ([0, 3, 4], [2, 0])}[max_size]
    assert (gs.tolist(), pre.tolist()) == want


def test_prefix_stops_before_each_members_last_token():
    tables = np.array([[1, 2, 3], [1, 2, 3], [1, 2, 3]])
    # lengths 33, 32, 48: whole blocks before the last token are 2, 1, 2
    gs, pre = ops.prefix_groups(tables, np.array([33, 32, 48]), 8)
    assert gs.tolist() == [0, 3] and pre.tolist() == [1]


def test_empty_and_unrelated_sequences_start_their_own_groups():
    tables = np.array([[1, 2], [1, 2], [3, 4], [5, 6]])
    gs, pre = ops.prefix_groups(tables, np.array([0, 20, 20, 20]), 4)
    assert gs.tolist() == [0, 1, 2, 3, 4] and pre.tolist() == [0, 0, 0, 0]


def _prefix_by_definition(tables, lens, gs):
    out = []
    for i in range(len(gs) - 1):
        rows = tables[gs[i]:gs[i + 1]]
        nblk = -(-int(lens[gs[i]:gs[i + 1]].max()) // 16)
        n = 0
        while n < nblk and all(r[n] == rows[0][n] for r in rows):
            n += 1
        out.append(n)
    return out


@pytest.mark.parametrize("equal_groups", [True, False])
def test_shared_table_prefix_matches_its_definition(palib, equal_groups):
    """Beams of three prompts reselected from parents for several steps (as
    beam search does), so groups share the prompt and tail blocks inherited
    from common ancestors: the helper's count equals the leading entries
    every member holds, for equal and unequal group sizes."""
    rng = np.random.Generator(np.random.PCG64(8))
    sizes = [4, 4, 4] if equal_groups else [4, 2, 3]
    a = ops.BlockAllocator(600, rng.permutation(600))
    ids, gs = [], [0]
    for g, n in enumerate(sizes):
        a.alloc_seq(10_000 + g, 32 * 16 + 7 * g)
        kids = list(range(len(ids), len(ids) + n))
        a.fork_seqs([10_000 + g] * n, kids)
        for k in kids:
            a.append_tokens(k, int(rng.integers(1, 60)), want_slots=False)
        ids += kids
        gs.append(len(ids))
    for step in range(12):
        par = [gs[g] + int(rng.integers(0, sizes[g])) - gs[g] for g in range(len(sizes)) for _ in range(sizes[g])]
        par = [gs[g] + p for g, p in zip([g for g in range(len(sizes)) for _ in range(sizes[g])], par)]
        a.reselect(ids, par)
        a.append_slots(ids)
        tables, lens = a.tables(ids, 80)
        got = ops.shared_table_prefix(tables, lens, np.asarray(gs))
        assert got.tolist() == _prefix_by_definition(tables, lens, gs)
