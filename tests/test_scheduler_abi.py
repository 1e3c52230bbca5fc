"""The C++ scheduler (pa_sched_*) against the oracle's scheduler model:
identical decisions -- items, slots, retirements, swap pairs, drops -- at
every step of the hand-derived traces and of random arrival traces.  Needs
only the host library (no GPU)."""
import random

import pytest

from oracle.allocator import blocks_for
from oracle.scheduler import Scheduler as OSched
from paged_kv_cache_191_gb300 import ops
from tests.libfixture import palib  # noqa: F401
from tests.scheduler_trace import replay

pytestmark = pytest.mark.usefixtures("palib")


class _CAdapter:
    def __init__(self, nb, mb, mt, hb):
        self.s = ops.Scheduler(nb, mb, mt, hb)

    def add(self, rid, prompt, max_new):
        self.s.add(rid, prompt, max_new)

    def step(self):
        return self.s.step()

    def idle(self):
        return self.s.idle()


def test_hand_derived_traces():
    def check(ok, where, got, want):
        assert ok, f"{where}: got {got!r}, want {want!r}"
    replay(_CAdapter, check)


@pytest.mark.parametrize("seed", range(60))
def test_random_traces_match_the_oracle(seed):
    rnd = random.Random(1000 + seed)
    nb = rnd.choice([6, 12, 40, 200])
    mb, mt, hb = rnd.choice([1, 2, 4, 8, 32]), rnd.choice([8, 16, 64, 256, 2048]), rnd.choice([0, 3, 16, 64])
    order = rnd.sample(range(nb), nb)
    c, o = ops.Scheduler(nb, mb, mt, hb, order), OSched(nb, mb, mt, hb, order)
    n_req = rnd.randint(5, 40)
    arrivals = sorted(rnd.randint(0, 80) for _ in range(n_req))
    specs = []
    for i in range(n_req):
        while True:
            p, m = rnd.randint(1, 300), rnd.randint(1, 60)
            if blocks_for(p + m) <= nb:
                break
        specs.append((arrivals[i], 7 * i + 3, p, m))
    it = 0
    while True:
        for t, rid, p, m in specs:
            if t == it:
                c.add(rid, p, m)
                o.add(rid, p, m)
        got = c.step()
        r = o.step()
        want = (r.items, r.finished, r.swap_out, r.swap_in, r.recomputed)
        assert got == want, f"step {it}"
        it += 1
        if o.idle() and it > arrivals[-1]:
            break
        assert it < 20000
    assert c.idle()
    w, run, sw, free, hfree = c.stats()
    assert (free, hfree) == (nb, hb)


def test_errors():
    s = ops.Scheduler(4, 2, 64, 0)
    with pytest.raises(ops.PagedKVError):
        s.add(1, 60, 5)
    with pytest.raises(ops.PagedKVError):
        s.add(2, 0, 1)
    s.add(3, 10, 1)
    with pytest.raises(ops.PagedKVError):
        s.add(3, 10, 1)
    with pytest.raises(ops.PagedKVError):
        ops.Scheduler(4, 0, 64, 0)
