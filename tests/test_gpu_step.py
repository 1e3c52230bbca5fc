"""Whole decode steps on the GPU against the oracle, step by step.

Each step runs the path the benchmark times: the block manager (C++) appends
one slot per sequence -- copy-on-write when a shared partial block is
written -- then pa_copy_blocks, pa_cache_write and pa_decode run on the
device.  The oracle runs the same steps with its own block-manager model,
cache write, block copy and attention.  Slots, tables and copy pairs must be
identical, caches bit-identical, outputs within the attention tolerance.

Two flows: a growing batch (sequences admitted at their lengths, one token
per step, the LLaMA-7B-shaped workload at reduced batch), and shared-prefix
beam search (groups of beams forked from one prompt, beams reselected from
parents every step, so siblings share partially filled blocks and appends
trigger copy-on-write).
"""
import numpy as np
import pytest
import torch

from oracle.allocator import BlockAllocator as OAlloc
from oracle.attention import paged_decode
from oracle.cache_ops import cache_write as o_write, copy_blocks as o_copy
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, assert_close, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


class Pair:
    """The C++ block manager and the oracle model, driven in lockstep."""

    def __init__(self, num_blocks, order):
        self.c = ops.BlockAllocator(num_blocks, order)
        self.o = OAlloc(num_blocks, order)

    def both(self, name, *args):
        a = getattr(self.c, name)(*args)
        b = getattr(self.o, name)(*args)
        return a, b


def _device_state(w_pool_k, w_pool_v):
    return w_pool_k.to(DEV), w_pool_v.to(DEV)


def _run_step(al, ids, kc, vc, okc, ovc, q, nk, nv, scale, cap):
    """One step on both sides; returns (gpu out, oracle out, n copies)."""
    slots, pairs = al.c.append_slots(ids)
    want = al.o.append_slots(ids)
    assert slots == [x[0] for x in want]
    assert pairs == [(x[1], x[2]) for x in want if x[1] >= 0]
    tables, lens = al.c.tables(ids, cap)
    for i, s in enumerate(ids):
        tab, n = al.o.table(s)
        assert list(tables[i][:len(tab)]) == tab and lens[i] == n
    if pairs:
        ops.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int64, device=DEV))
        okc, ovc, _, _ = o_copy(okc, ovc, pairs)
    ops.cache_write(nk.to(DEV), nv.to(DEV), torch.tensor(slots, device=DEV), kc, vc)
    okc, ovc, _, _ = o_write(np_exact(nk), np_exact(nv), np.array(slots), okc, ovc)
    out = ops.decode(q.to(DEV), kc, vc, torch.from_numpy(tables).to(DEV), torch.from_numpy(lens).to(DEV),
                     int(lens.max()), scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = paged_decode(np_exact(q), okc, ovc, tables, lens, scale)
    return out.cpu().numpy(), ref, okc, ovc, len(pairs)


def test_growing_batch_steps():
    w = W.config_llama7b(B=6)
    al = Pair(w.num_blocks + 64, list(w.free_order) + list(range(w.num_blocks, w.num_blocks + 64)))
    kp = torch.cat([w.k_pool, torch.zeros((64,) + tuple(w.k_pool.shape[1:]), dtype=w.k_pool.dtype)])
    vp = torch.cat([w.v_pool, torch.zeros((64,) + tuple(w.v_pool.shape[1:]), dtype=w.v_pool.dtype)])
    ids = list(range(w.B))
    for b in ids:
        al.both("alloc_seq", b, int(w.context_lens[b]) - 1)
    kc, vc = kp.to(DEV), vp.to(DEV)
    okc, ovc = np_exact(kp), np_exact(vp)
    cap = -(-(int(w.context_lens.max()) + 8) // 16)
    rng = W.rng_for(5)
    for step in range(3):
        nk = W.randn(rng, (w.B, w.Hkv, w.D), torch.float16)
        nv = W.randn(rng, (w.B, w.Hkv, w.D), torch.float16)
        out, ref, okc, ovc, ncow = _run_step(al, ids, kc, vc, okc, ovc, w.q, nk, nv, w.scale, cap)
        assert ncow == 0
        assert_close(out, ref, TOL["f16"], f"growing step {step}")
    assert np.array_equal(np_exact(kc), okc) and np.array_equal(np_exact(vc), ovc)


@pytest.mark.parametrize("prompt", [40, 64])
def test_shared_prefix_beam_steps(prompt):
    groups, beams, H, D = 3, 4, 8, 128
    rng = W.rng_for(11 + prompt)
    nb = 200
    order = rng.permutation(nb).astype(np.int64)
    al = Pair(nb, order)
    kp = W.randn(rng, (nb, H, 16, D), torch.float16)
    vp = W.randn(rng, (nb, H, 16, D), torch.float16)
    kc, vc = kp.to(DEV), vp.to(DEV)
    okc, ovc = np_exact(kp), np_exact(vp)
    nxt = 1000
    roots = []
    for g in range(groups):
        al.both("alloc_seq", 900 + g, prompt)
        roots.append(900 + g)
    ids = []
    tails = rng.integers(1, 30, size=(groups, beams))
    for g in range(groups):
        for i in range(beams):
            al.both("fork", roots[g], nxt)
            got, want = al.both("append_tokens", nxt, int(tails[g][i]))
            assert got == (want[0], want[1])
            if want[1][0] >= 0:  # a tail that starts in the shared partial prompt block
                ops.copy_blocks(kc, vc, torch.tensor([want[1]], dtype=torch.int64, device=DEV))
                okc, ovc, _, _ = o_copy(okc, ovc, [want[1]])
            ids.append(nxt)
            nxt += 1
    al.both("free_seqs", roots)
    cap = -(-(prompt + 40 + 8) // 16)
    q = W.randn(rng, (groups * beams, H, D), torch.float16)
    total_cow = 0
    for step in range(4):
        parents = rng.integers(0, beams, size=(groups, beams))
        new = list(range(nxt, nxt + groups * beams))
        nxt += groups * beams
        if step % 2:  # reselection by fork + release ...
            par = [ids[g * beams + int(parents[g][j])] for g in range(groups) for j in range(beams)]
            al.both("fork_seqs", par, new)
            al.both("free_seqs", ids)
            ids = new
        else:         # ... or in place
            al.both("reselect", ids, [g * beams + int(parents[g][j]) for g in range(groups) for j in range(beams)])
        nk = W.randn(rng, (len(ids), H, D), torch.float16)
        nv = W.randn(rng, (len(ids), H, D), torch.float16)
        out, ref, okc, ovc, ncow = _run_step(al, ids, kc, vc, okc, ovc, q, nk, nv, 1 / np.sqrt(D), cap)
        total_cow += ncow
        assert_close(out, ref, TOL["f16"], f"beam step {step}")
    assert total_cow > 0, "the workload is meant to exercise copy-on-write"
    assert np.array_equal(np_exact(kc), okc) and np.array_equal(np_exact(vc), ovc)
    c_tot, c_free, c_rc = al.c.stats()
    assert (c_free, c_rc) == (len(al.o.free), al.o.refcount)
