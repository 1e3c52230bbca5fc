"""Pins for the oracle's continuous-batching scheduler.

(a) three hand-derived traces in tests/golden (plain admission and retirement
with chunked prefill; preemption by swap with the tie rule, the delayed
swap-in and the block placement; preemption by recompute);
(b) properties on random arrival traces, after every step: the block manager
and host-pool invariants, batch and token budgets, each request's cache
holding exactly its progress, admissions in arrival order, every slot
written once per step; the preemption victim (the largest holder when it
fits the host pool, else the smallest is dropped); and liveness: every
request finishes, with its cache holding prompt + max_new - 1 tokens at the
end, and the pools come back whole.
"""
import random

import pytest

from oracle.allocator import InvalidOp, blocks_for
from oracle.scheduler import Scheduler, DECODE, PREFILL
from tests.scheduler_trace import replay


class _Adapter:
    def __init__(self, nb, mb, mt, hb):
        self.s = Scheduler(nb, mb, mt, hb)

    def add(self, rid, prompt, max_new):
        self.s.add(rid, prompt, max_new)

    def step(self):
        r = self.s.step()
        self.s.check_invariants()
        return r.items, r.finished, r.swap_out, r.swap_in, r.recomputed

    def idle(self):
        return self.s.idle()


def test_hand_derived_traces():
    def check(ok, where, got, want):
        assert ok, f"{where}: got {got!r}, want {want!r}"
    replay(_Adapter, check)


def test_refuses_requests_that_cannot_complete():
    s = Scheduler(4, 2, 64, 0)
    with pytest.raises(InvalidOp):
        s.add(1, 60, 5)           # 65 tokens need 5 blocks of 4
    with pytest.raises(InvalidOp):
        s.add(2, 0, 5)
    s.add(3, 60, 4)
    with pytest.raises(InvalidOp):
        s.add(3, 1, 1)            # id in use


def run_trace(seed, steps_max=5000):
    rnd = random.Random(seed)
    nb = rnd.choice([6, 12, 40])
    s = Scheduler(nb, rnd.choice([1, 2, 4, 8]), rnd.choice([8, 16, 64, 256]), rnd.choice([0, 3, 16, 64]),
                  free_order=rnd.sample(range(nb), nb))
    n_req = rnd.randint(5, 25)
    arrivals = sorted(rnd.randint(0, 60) for _ in range(n_req))
    specs = {}
    for i in range(n_req):
        while True:
            prompt, max_new = rnd.randint(1, 120), rnd.randint(1, 40)
            if blocks_for(prompt + max_new) <= nb:
                break
        specs[100 + i] = (arrivals[i], prompt, max_new)
    outputs = {rid: 0 for rid in specs}
    finished = []
    admitted_order = []
    it = 0
    while True:
        for rid, (t, p, m) in specs.items():
            if t == it:
                s.add(rid, p, m)
        res = s.step()
        s.check_invariants()
        # budgets
        assert len(s.running) <= s.max_batch
        n_dec = sum(1 for _, k, _, _ in res.items if k == "decode")
        n_pre = sum(len(sl) for _, k, _, sl in res.items if k == "prefill")
        assert n_pre <= max(0, s.max_tokens - n_dec)
        # every slot written once this step
        slots = [x for _, _, _, sl in res.items for x in sl]
        assert len(slots) == len(set(slots))
        for rid, kind, start, sl in res.items:
            if kind == "prefill" and start == 0:
                admitted_order.append(rid)
            if kind == "decode":
                outputs[rid] += 1
        for rid in res.recomputed:
            outputs[rid] = 0
        for rid in res.finished:
            finished.append(rid)
        it += 1
        if s.idle() and it > max(arrivals):
            break
        assert it < steps_max, "scheduler made no progress"
    assert sorted(finished) == sorted(specs)
    assert len(s.alloc.free) == nb and len(s.host_free) == s.host_total
    return s, specs, admitted_order


@pytest.mark.parametrize("seed", range(40))
def test_random_traces(seed):
    run_trace(seed)


def test_admission_is_first_come_first_served_without_preemption():
    for seed in range(30):
        rnd = random.Random(seed)
        s = Scheduler(200, 4, 64, 0)
        ids = list(range(12))
        for i in ids:
            s.add(i, rnd.randint(1, 100), rnd.randint(1, 30))
        first_chunk = []
        while not s.idle():
            res = s.step()
            assert not res.recomputed and not res.swap_out
            first_chunk += [rid for rid, k, st, _ in res.items if k == "prefill" and st == 0]
        assert first_chunk == ids


def test_each_request_gets_its_prompt_and_outputs_exactly():
    """Cache tokens at retirement = prompt + max_new - 1 (the last output's
    K/V is never appended); outputs produced = max_new."""
    for seed in range(20):
        rnd = random.Random(seed)
        s = Scheduler(30, 3, 32, 8)
        want = {}
        for i in range(10):
            p, m = rnd.randint(1, 150), rnd.randint(1, 60)
            if blocks_for(p + m) > 30:
                continue
            s.add(i, p, m)
            want[i] = (p, m)
        seen_tokens = {i: 0 for i in want}
        while not s.idle():
            res = s.step()
            for rid, k, st, sl in res.items:
                assert s.reqs[rid].ctx() == st + len(sl)
                seen_tokens[rid] = st + len(sl)
            for rid in res.recomputed:
                seen_tokens[rid] = 0
            for rid in res.finished:
                p, m = want[rid]
                assert seen_tokens[rid] == p + m - 1, (rid, seen_tokens[rid], p, m)


def _until_preemption(s, limit=60):
    for _ in range(limit):
        held = {r.id: len(s.alloc.tables[r.id]) for r in s.running}
        res = s.step()
        if res.swap_out or res.recomputed:
            return held, res
    pytest.fail("no preemption happened")


def test_swap_takes_the_largest_holder():
    s = Scheduler(8, 3, 200, 100)
    s.add(1, 40, 60)   # 3 blocks after its prefill
    s.add(2, 60, 60)   # 4 blocks
    s.step()
    held, res = _until_preemption(s)
    assert len(res.swap_out) == max(held.values())
    victim = [rid for rid in held if rid not in {r.id for r in s.running}]
    assert victim == [max(held, key=lambda k: (held[k], s.reqs[k].arrival))]
    assert [h for _, h in res.swap_out] == list(range(len(res.swap_out)))  # host free list front


def test_drop_takes_the_smallest_holder_when_the_host_pool_is_full():
    s = Scheduler(8, 3, 200, 0)
    s.add(1, 40, 60)
    s.add(2, 60, 60)
    s.step()
    held, res = _until_preemption(s)
    assert not res.swap_out
    assert res.recomputed == [min(held, key=lambda k: (held[k], -s.reqs[k].arrival))]
