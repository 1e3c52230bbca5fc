"""The C++ block manager behind the C ABI, held to the hand-derived trace and
compared operation by operation with the oracle model (bit-exact slots,
tables, copy-on-write pairs, free-list order and refcounts).  Host only."""
import random

import numpy as np
import pytest

from oracle.allocator import BlockAllocator as OracleAlloc, OutOfBlocks as OOOM, UnknownSeq, InvalidOp
from paged_kv_cache_191_gb300 import ops
from tests.allocator_trace import replay
from tests.libfixture import palib  # noqa: F401


class _Adapter:
    def __init__(self, pool):
        self.a = ops.BlockAllocator(pool)

    def _run(self, fn, *args):
        try:
            r = fn(*args)
            return "ok" if r is None else ("ok", r)
        except ops.OutOfBlocks:
            return "oom"
        except ops.UnknownSequence:
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
        return self.a.free_list()

    def utilization(self):
        return self.a.utilization()


def test_hand_derived_trace(palib):
    def check(ok, op, args, got, want):
        assert ok, f"{op} {args}: got {got!r}, want {want!r}"
    replay(_Adapter, check)


def _same_state(c, o):
    assert c.free_list() == list(o.free)
    tot, fr, rc = c.stats()
    assert (tot, fr) == (o.total, len(o.free)) and rc == o.refcount
    for s in o.tables:
        assert c.table(s) == o.table(s)


@pytest.mark.parametrize("seed", range(10))
def test_matches_oracle_model_on_random_operations(palib, seed):
    rnd = random.Random(100 + seed)
    pool = rnd.choice([8, 24, 64])
    order = rnd.sample(range(pool), pool)
    c, o = ops.BlockAllocator(pool, order), OracleAlloc(pool, order)
    live, nxt = [], 1
    for _ in range(300):
        op = rnd.choice(["alloc", "append", "append", "batch", "fork", "free", "bad",
                         "tokens", "forks", "frees", "reselect"])
        if op == "alloc":
            n = rnd.randint(0, 50)
            exp = None
            try:
                o.alloc_seq(nxt, n)
            except OOOM as e:
                exp = e
            if exp:
                with pytest.raises(ops.OutOfBlocks):
                    c.alloc_seq(nxt, n)
            else:
                c.alloc_seq(nxt, n)
                live.append(nxt)
                nxt += 1
        elif op == "append" and live:
            s = rnd.choice(live)
            try:
                want = o.append_slot(s)
            except OOOM:
                with pytest.raises(ops.OutOfBlocks):
                    c.append_slot(s)
            else:
                assert c.append_slot(s) == want
        elif op == "batch" and live:
            seqs = rnd.sample(live, rnd.randint(1, min(5, len(live))))
            try:
                want = o.append_slots(seqs)
            except OOOM:
                with pytest.raises(ops.OutOfBlocks):
                    c.append_slots(seqs)
            else:
                slots, pairs = c.append_slots(seqs)
                assert slots == [w[0] for w in want]
                assert pairs == [(w[1], w[2]) for w in want if w[1] >= 0]
        elif op == "fork" and live:
            p = rnd.choice(live)
            o.fork(p, nxt)
            c.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        elif op == "free" and live:
            s = live.pop(rnd.randrange(len(live)))
            o.free_seq(s)
            c.free_seq(s)
        elif op == "tokens" and live:
            sq, n = rnd.choice(live), rnd.randint(0, 40)
            try:
                want = o.append_tokens(sq, n)
            except OOOM:
                with pytest.raises(ops.OutOfBlocks):
                    c.append_tokens(sq, n)
            else:
                got = c.append_tokens(sq, n)
                assert got[0] == want[0] and got[1] == want[1]
        elif op == "forks" and live:
            k = rnd.randint(1, 4)
            parents, children = [], []
            for _ in range(k):  # a child may be a later parent
                parents.append(rnd.choice(live + children))
                children.append(nxt)
                nxt += 1
            o.fork_seqs(parents, children)
            c.fork_seqs(parents, children)
            live.extend(children)
        elif op == "frees" and live:
            k = rnd.randint(1, min(4, len(live)))
            ids = rnd.sample(live, k)
            o.free_seqs(ids)
            c.free_seqs(ids)
            for i in ids:
                live.remove(i)
        elif op == "reselect" and live:
            k = rnd.randint(1, min(6, len(live)))
            ids = rnd.sample(live, k)
            par = [rnd.randrange(k) for _ in range(k)]
            o.reselect(ids, par)
            c.reselect(ids, par)
        elif op == "bad":
            with pytest.raises(ops.UnknownSequence):
                c.append_slot(10 ** 9)
            with pytest.raises(ops.UnknownSequence):
                c.free_seq(10 ** 9)
            with pytest.raises(ops.UnknownSequence):
                c.fork_seqs([10 ** 9], [nxt])
            with pytest.raises(ops.UnknownSequence):
                c.append_tokens(10 ** 9, 3)
            if live:
                with pytest.raises(ops.PagedKVError):
                    c.free_seqs([live[0], live[0]])
                with pytest.raises(ops.PagedKVError):
                    c.fork_seqs([live[0]], [live[0]])
                with pytest.raises(ops.PagedKVError):
                    c.alloc_seq(live[0], 1)
                with pytest.raises(ops.PagedKVError):
                    c.append_slots([live[0], live[0]])
        _same_state(c, o)


def test_block_tables_are_padded_and_report_lengths(palib):
    a = ops.BlockAllocator(10)
    a.alloc_seq(7, 33)
    a.alloc_seq(9, 0)
    tab, lens = a.tables([7, 9], cap=4)
    assert tab.tolist() == [[0, 1, 2, -1], [-1, -1, -1, -1]]
    assert lens.tolist() == [33, 0]
    with pytest.raises(ops.PagedKVError):
        a.tables([7], cap=2)


def test_create_rejects_bad_pool(palib):
    with pytest.raises(ops.PagedKVError):
        ops.BlockAllocator(0)
    with pytest.raises(ops.PagedKVError):
        ops.BlockAllocator(3, free_order=[0, 0, 1])
