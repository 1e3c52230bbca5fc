"""Replay of the hand-derived block-manager trace in tests/golden.

Shared by the oracle-allocator test and the C-ABI allocator test: it only
parses the fixture and drives a small adapter interface, so that both
implementations are held to the same hand-derived expectations.
"""
import os
from fractions import Fraction

TRACE = os.path.join(os.path.dirname(__file__), "golden", "allocator_trace.txt")


def load_trace():
    ops = []
    for line in open(TRACE):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("pool"):
            ops.append(("pool", int(line.split()[1]), None))
            continue
        lhs, rhs = [x.strip() for x in line.split("->")]
        ops.append((lhs.split()[0], lhs.split()[1:], rhs))
    return ops


def replay(make, check):
    """make(pool) -> adapter with alloc/append/fork/free_seq/table/free_list/
    utilization returning ("ok"|"oom"|"notfound", payload)."""
    ids = {}

    def sid(name):
        return ids.setdefault(name, len(ids) + 1)

    a = None
    for op, args, want in load_trace():
        if op == "pool":
            a = make(args)
            continue
        if op == "alloc":
            got = a.alloc(sid(args[0]), int(args[1]))
            check(got == want, op, args, got, want)
        elif op == "append":
            status, payload = a.append(sid(args[0]))
            if status == "ok":
                slot, src, dst = payload
                got = f"slot={slot} cow={src},{dst}"
            else:
                got = status
            check(got == want, op, args, got, want)
        elif op == "fork":
            got = a.fork(sid(args[0]), sid(args[1]))
            check(got == want, op, args, got, want)
        elif op == "free_seq":
            got = a.free_seq(sid(args[0]))
            check(got == want, op, args, got, want)
        elif op == "table":
            blocks, n = a.table(sid(args[0]))
            got = ",".join(str(b) for b in blocks) + f" n={n}"
            check(got == want, op, args, got, want)
        elif op == "free":
            got = ",".join(str(b) for b in a.free_list())
            check(got == want, op, args, got, want)
        elif op == "utilization":
            num, den = want.split("/")
            check(Fraction(a.utilization()).limit_denominator(1000) == Fraction(int(num), int(den)),
                  op, args, a.utilization(), want)
        else:
            raise ValueError(op)
