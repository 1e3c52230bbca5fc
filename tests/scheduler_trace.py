"""Replay of tests/golden/scheduler_trace.txt against a scheduler adapter.

An adapter is built as make(num_blocks, max_batch, max_tokens, host_blocks)
and offers add(id, prompt, max_new), step() -> (items, finished, swap_out,
swap_in, recomputed) with items as (id, kind, start, slots), and idle().
"""
import os

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scheduler_trace.txt")


def _slots(text):
    out = []
    for part in filter(None, text.split(",")):
        a, _, b = part.partition("-")
        out.extend(range(int(a), int(b or a) + 1))
    return out


def _pairs(text):
    return [tuple(int(x) for x in p.split(">")) for p in filter(None, text.split(","))]


def _ids(text):
    return [int(x) for x in filter(None, text.split(","))]


def parse_step(line):
    fields = dict(f.split("=", 1) for f in line.split()[1:])
    items = []
    for it in filter(None, fields["items"].split(";")):
        rid, kind, start, slots = it.split(":")
        items.append((int(rid), kind, int(start), _slots(slots)))
    return items, _ids(fields["finished"]), _pairs(fields["out"]), _pairs(fields["in"]), _ids(fields["rec"])


def replay(make, check):
    """Run every scenario; check(ok, where, got, want) reports each step."""
    sched, name, n = None, None, 0
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            op = line.split()[0]
            if op == "scenario":
                _, name, nb, mb, mt, hb = line.split()
                sched, n = make(int(nb), int(mb), int(mt), int(hb)), 0
            elif op == "add":
                _, rid, prompt, max_new = line.split()
                sched.add(int(rid), int(prompt), int(max_new))
            elif op == "step":
                want = parse_step(line)
                got = sched.step()
                check(tuple(got) == want, f"{name} step {n}", got, want)
                n += 1
            elif op == "idle":
                check(sched.idle(), f"{name} idle", sched.idle(), True)
