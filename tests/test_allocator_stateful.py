"""Property-based (hypothesis) state machine over the block manager.

The oracle model and the C++ block manager behind the C ABI are driven in
lockstep by operation sequences that hypothesis generates and shrinks.  After
every operation:

* both sides agree bit for bit (free-list order, refcounts, tables, token
  counts, returned slots and copy-on-write pairs, error kinds);
* the oracle's invariants hold (free + distinct referenced = total; refcount =
  number of tables holding the block; the free list has no duplicate and no
  referenced block; table length = ceil(tokens / 16));
* utilisation = used / total, the figure the continuous-batching article's
  block manager reports ("大模型推理引擎优化：KV Cache 与连续批处理", section 三);
* a failed operation (out of blocks, unknown sequence) leaves the state
  unchanged on both sides.

Host only: no GPU.
"""
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, settings, strategies as st  # noqa: E402
from hypothesis.stateful import RuleBasedStateMachine, initialize, invariant, precondition, rule  # noqa: E402

from oracle.allocator import BlockAllocator as OracleAlloc, OutOfBlocks as OOOM, UnknownSeq  # noqa: E402
from paged_kv_cache_191_gb300 import ops  # noqa: E402
from tests.libfixture import palib  # noqa: E402,F401


def _snapshot(o):
    return (list(o.free), list(o.refcount), {s: (list(t), o.ntokens[s]) for s, t in o.tables.items()})


class BlockManagerMachine(RuleBasedStateMachine):
    def __init__(self):
        super().__init__()
        self.o = self.c = None
        self.live, self.next_id = [], 1

    @initialize(pool=st.sampled_from([4, 9, 16, 33]), data=st.data())
    def make(self, pool, data):
        order = data.draw(st.permutations(list(range(pool))))
        self.o, self.c = OracleAlloc(pool, order), ops.BlockAllocator(pool, order)

    def _fresh(self):
        s = self.next_id
        self.next_id += 1
        return s

    def _expect_same_failure(self, o_call, c_call):
        """Run o_call; on a refusal, check c_call refuses the same way and
        that neither side changed.  Returns o_call's result or None."""
        before = _snapshot(self.o)
        try:
            return True, o_call()
        except OOOM:
            kind = ops.OutOfBlocks
        except UnknownSeq:
            kind = ops.UnknownSequence
        assert _snapshot(self.o) == before, "oracle changed state on a refused operation"
        with pytest.raises(kind):
            c_call()
        return False, None

    @rule(n=st.integers(0, 70))
    def alloc(self, n):
        s = self._fresh()
        ok, _ = self._expect_same_failure(lambda: self.o.alloc_seq(s, n), lambda: self.c.alloc_seq(s, n))
        if ok:
            self.c.alloc_seq(s, n)
            self.live.append(s)

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def append(self, data):
        s = data.draw(st.sampled_from(self.live))
        ok, want = self._expect_same_failure(lambda: self.o.append_slot(s), lambda: self.c.append_slot(s))
        if ok:
            assert self.c.append_slot(s) == want

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def append_batch(self, data):
        seqs = data.draw(st.lists(st.sampled_from(self.live), min_size=1, max_size=6, unique=True))
        ok, want = self._expect_same_failure(lambda: self.o.append_slots(seqs), lambda: self.c.append_slots(seqs))
        if ok:
            slots, pairs = self.c.append_slots(seqs)
            assert slots == [w[0] for w in want]
            assert pairs == [(w[1], w[2]) for w in want if w[1] >= 0]

    @precondition(lambda self: self.live)
    @rule(data=st.data(), n=st.integers(0, 40))
    def append_tokens(self, data, n):
        s = data.draw(st.sampled_from(self.live))
        ok, want = self._expect_same_failure(lambda: self.o.append_tokens(s, n), lambda: self.c.append_tokens(s, n))
        if ok:
            got = self.c.append_tokens(s, n)
            assert got[0] == want[0] and got[1] == want[1]

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def fork(self, data):
        p, child = data.draw(st.sampled_from(self.live)), self._fresh()
        self.o.fork(p, child)
        self.c.fork(p, child)
        self.live.append(child)

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def free(self, data):
        s = data.draw(st.sampled_from(self.live))
        self.live.remove(s)
        self.o.free_seq(s)
        self.c.free_seq(s)

    @precondition(lambda self: self.live)
    @rule(data=st.data())
    def reselect(self, data):
        seqs = data.draw(st.lists(st.sampled_from(self.live), min_size=1, max_size=6, unique=True))
        par = data.draw(st.lists(st.integers(0, len(seqs) - 1), min_size=len(seqs), max_size=len(seqs)))
        self.o.reselect(seqs, par)
        self.c.reselect(seqs, par)

    @rule()
    def unknown_sequence(self):
        ghost = 10 ** 9
        self._expect_same_failure(lambda: self.o.append_slot(ghost), lambda: self.c.append_slot(ghost))
        self._expect_same_failure(lambda: self.o.free_seq(ghost), lambda: self.c.free_seq(ghost))

    @invariant()
    def agree_and_hold(self):
        if self.o is None:
            return
        o, c = self.o, self.c
        o.check_invariants()
        assert c.free_list() == list(o.free)
        tot, fr, rc = c.stats()
        assert (tot, fr) == (o.total, len(o.free)) and rc == o.refcount
        used = sum(1 for r in o.refcount if r > 0)
        assert o.utilization() == pytest.approx(used / o.total, abs=0)
        assert c.utilization() == pytest.approx(used / o.total, rel=1e-12)
        for s in self.live:
            assert c.table(s) == o.table(s)


def test_block_manager_state_machine(palib):
    BlockManagerMachine.TestCase.settings = settings(
        max_examples=60, stateful_step_count=40, deadline=None,
        suppress_health_check=[HealthCheck.too_slow, HealthCheck.data_too_large])
    hypothesis.stateful.run_state_machine_as_test(BlockManagerMachine, settings=BlockManagerMachine.TestCase.settings)
