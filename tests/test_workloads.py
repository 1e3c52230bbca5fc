"""The seeded input recipe: pool size, tables taken in order from a permuted
pool (what a FIFO block manager with that free list hands out), storage-dtype
rounding of N(0, 1) draws, and determinism by seed.  Host only, small shapes."""
import math

import numpy as np
import torch

from paged_kv_cache_191_gb300 import workloads as W
from oracle.allocator import BlockAllocator


def test_tables_are_what_a_fifo_block_manager_hands_out():
    lens = [5, 17, 32, 47, 1, 0, 160]
    w = W.make_decode("t", 7, len(lens), 4, 2, 64, "f16", lens)
    demand = sum(-(-n // 16) for n in lens)
    assert w.num_blocks == max(math.ceil(1.2 * demand), demand, 1)
    assert sorted(w.free_order.tolist()) == list(range(w.num_blocks))
    alloc = BlockAllocator(w.num_blocks, w.free_order)
    for b, n in enumerate(lens):
        alloc.alloc_seq(b, n)
        tab, ntok = alloc.table(b)
        nb = -(-n // 16)
        assert ntok == n and tab == w.block_tables[b, :nb].tolist()
        assert (w.block_tables[b, nb:] == -1).all()
    assert w.block_tables.shape == (len(lens), max(-(-n // 16) for n in lens))


def test_draws_are_seeded_and_rounded_once():
    a = W.make_decode("t", 11, 3, 8, 2, 128, "bf16", [40, 3, 100])
    b = W.make_decode("t", 11, 3, 8, 2, 128, "bf16", [40, 3, 100])
    c = W.make_decode("t", 12, 3, 8, 2, 128, "bf16", [40, 3, 100])
    for name in ("q", "k_pool", "v_pool", "new_k", "new_v"):
        ta, tb, tc = getattr(a, name), getattr(b, name), getattr(c, name)
        assert ta.dtype == torch.bfloat16
        assert torch.equal(ta, tb) and not torch.equal(ta, tc)
    assert np.array_equal(a.free_order, b.free_order)
    # the first draw after the permutation is q, N(0, 1) in float32 rounded once
    rng = W.rng_for(11)
    rng.permutation(a.num_blocks)
    q32 = rng.standard_normal(size=(3, 8, 128), dtype=np.float32)
    assert torch.equal(a.q, torch.from_numpy(q32).to(torch.bfloat16))
    assert abs(float(a.k_pool.float().mean())) < 0.05 and abs(float(a.k_pool.float().std()) - 1) < 0.05
    assert a.scale == 1 / math.sqrt(128)


def test_tiny_workload_recipe():
    w = W.config_tiny()
    assert (w.B, w.Hq, w.Hkv, w.D, w.kv_dtype) == (4, 4, 4, 64, "f16")
    assert w.context_lens.tolist() == [5, 17, 32, 47] and w.num_blocks == 32
    assert w.k_pool.shape == (32, 4, 16, 64) and w.q.dtype == torch.float16
