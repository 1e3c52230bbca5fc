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
