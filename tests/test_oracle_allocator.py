"""Pins for the oracle's block manager.

(a) the hand-derived trace in tests/golden (FIFO free list, ceil(n/16)
blocks, check-before-mutate, utilisation, copy-on-write on append);
(b) invariants after every operation of random operation sequences:
free + |referenced| = total, refcount(b) = number of tables holding b, the
free list has no duplicates and no referenced block, len(table) =
ceil(n/16), and a failed operation leaves the state unchanged.
"""
import copy

import pytest

from oracle.allocator import BlockAllocator, OutOfBlocks, UnknownSeq, InvalidOp, blocks_for
from tests.allocator_trace import replay


class _OracleAdapter:
    def __init__(self, pool):
        self.a = BlockAllocator(pool)

    def _run(self, fn, *args):
        try:
            r = fn(*args)
            return "ok" if r is None else ("ok", r)
        except OutOfBlocks:
            return "oom"
        except UnknownSeq:
            return "notfound"

    def alloc(self, s, n):
        return self._run(self.a.alloc_seq, s, n)

    def append(self, s):
        r = self._run(self.a.append_slot, s)
        return r if isinstance(r, tuple) else (r, None)

    def fork(self, p, c):
        return self._run(self.a.fork, p, c)

    def free_seq(self, s):
        return self._run(self.a.free_seq, s)

    def table(self, s):
        return self.a.table(s)

    def free_list(self):
        return list(self.a.free)

    def utilization(self):
        return self.a.utilization()


def test_hand_derived_trace():
    def check(ok, op, args, got, want):
        assert ok, f"{op} {args}: got {got!r}, want {want!r}"
    replay(_OracleAdapter, check)


def test_blocks_for_is_ceiling_of_sixteenths():
    assert [blocks_for(n) for n in (0, 1, 15, 16, 17, 32, 33)] == [0, 1, 1, 1, 2, 2, 3]


def _state(a):
    return (list(a.free), list(a.refcount), copy.deepcopy(a.tables), dict(a.ntokens))


def _random_ops(rng_seed, n_ops=400, pool=24):
    import random
    rnd = random.Random(rng_seed)
    a = BlockAllocator(pool, free_order=rnd.sample(range(pool), pool))
    live = []
    next_id = 1
    for _ in range(n_ops):
        op = rnd.choice(["alloc", "append", "append", "append", "fork", "free", "batch", "tokens",
                         "forks", "frees", "reselect"])
        before = _state(a)
        try:
            if op == "alloc":
                a.alloc_seq(next_id, rnd.randint(0, 40))
                live.append(next_id)
                next_id += 1
            elif op == "append" and live:
                slot, src, dst = a.append_slot(rnd.choice(live))
                assert slot >= 0
            elif op == "fork" and live:
                a.fork(rnd.choice(live), next_id)
                live.append(next_id)
                next_id += 1
            elif op == "free" and live:
                s = live.pop(rnd.randrange(len(live)))
                a.free_seq(s)
            elif op == "batch" and live:
                seqs = rnd.sample(live, min(len(live), rnd.randint(1, 4)))
                a.append_slots(seqs)
            elif op == "tokens" and live:
                sq = rnd.choice(live)
                n0 = a.ntokens[sq]
                slots, cow = a.append_tokens(sq, rnd.randint(0, 40))
                assert len(set(slots)) == len(slots)
                assert a.ntokens[sq] == n0 + len(slots)
            elif op == "forks" and live:
                kids = [next_id + i for i in range(rnd.randint(1, 3))]
                a.fork_seqs([rnd.choice(live) for _ in kids], kids)
                live.extend(kids)
                next_id += len(kids)
            elif op == "frees" and live:
                ids = rnd.sample(live, min(len(live), rnd.randint(1, 3)))
                a.free_seqs(ids)
                for i in ids:
                    live.remove(i)
            elif op == "reselect" and live:
                ids = rnd.sample(live, min(len(live), rnd.randint(1, 5)))
                par = [rnd.randrange(len(ids)) for _ in ids]
                want = [a.table(ids[p]) for p in par]
                a.reselect(ids, par)
                assert [a.table(s) for s in ids] == want
        except OutOfBlocks:
            assert _state(a) == before, "failed op changed the state"
        a.check_invariants()
        assert abs(a.utilization() - (a.total - len(a.free)) / a.total) < 1e-15
    return a


@pytest.mark.parametrize("seed", range(12))
def test_random_sequences_keep_invariants(seed):
    _random_ops(seed)


def test_slots_are_unique_among_live_tokens():
    import random
    rnd = random.Random(9)
    a = BlockAllocator(40)
    owner = {}
    for s in range(1, 5):
        a.alloc_seq(s, rnd.randint(1, 30))
    for _ in range(60):
        s = rnd.randint(1, 4)
        slot, src, dst = a.append_slot(s)
        assert a.refcount[slot // 16] == 1, "append wrote into a shared block"
        assert owner.get(slot, s) == s
        owner[slot] = s


def test_copy_on_write_when_forked_partial_block_is_appended():
    a = BlockAllocator(8)
    a.alloc_seq(1, 20)                  # blocks 0,1; block 1 holds 4 tokens
    a.fork(1, 2)
    assert a.refcount[:2] == [2, 2]
    slot, src, dst = a.append_slot(2)
    assert (src, dst) == (1, 2) and slot == 2 * 16 + 4
    assert a.table(2) == ([0, 2], 21) and a.refcount[:3] == [2, 1, 1]
    slot, src, dst = a.append_slot(1)   # the last sharer writes in place
    assert (src, dst) == (-1, -1) and slot == 16 + 4
    a.check_invariants()


def test_errors_leave_state_unchanged():
    a = BlockAllocator(3)
    a.alloc_seq(1, 32)
    before = _state(a)
    with pytest.raises(OutOfBlocks):
        a.alloc_seq(2, 17)
    with pytest.raises(InvalidOp):
        a.alloc_seq(1, 1)
    with pytest.raises(UnknownSeq):
        a.append_slot(9)
    with pytest.raises(InvalidOp):
        a.append_slots([1, 1])
    assert _state(a) == before
    a.alloc_seq(2, 16)
    before = _state(a)
    with pytest.raises(OutOfBlocks):
        a.append_slots([1, 2])          # both need a fresh block, none free
    assert _state(a) == before


def test_append_tokens_equals_repeated_appends():
    import random
    for seed in range(5):
        rnd = random.Random(seed)
        a, b = BlockAllocator(64), BlockAllocator(64)
        for al in (a, b):
            al.alloc_seq(1, 20)
            al.fork(1, 2)
        n = rnd.randint(1, 60)
        slots, cow = a.append_tokens(2, n)
        singles = [b.append_slot(2) for _ in range(n)]
        assert slots == [x[0] for x in singles]
        assert cow == next(((s, d) for _, s, d in singles if s >= 0), (-1, -1))
        assert a.tables == b.tables and list(a.free) == list(b.free) and a.refcount == b.refcount
