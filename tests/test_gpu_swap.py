"""Block swap between the GPU cache and a pinned host pool (preemption and
resume), against the oracle; and a whole preempt/resume round trip through the
block managers that must leave decode results bit-identical."""
import numpy as np
import pytest
import torch

from oracle.cache_ops import swap_blocks as o_swap
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import np_exact, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


@pytest.mark.parametrize("dt", ["f16", "bf16", "fp8", "int8"])
def test_swap_out_and_in(dt):
    rng = W.rng_for(21)
    N, NH, H, D = 64, 40, 8, 128
    if dt in ("fp8", "int8"):
        cdt, lo = (torch.int8, -128) if dt == "int8" else (torch.uint8, 0)
        gk = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
        gv = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
        gks, gvs = torch.rand((N, 16)), torch.rand((N, 16))
        hk = torch.zeros((NH, H, 16, D), dtype=cdt).pin_memory()
        hv = torch.zeros_like(hk).pin_memory()
        hks, hvs = torch.zeros((NH, 16)).pin_memory(), torch.zeros((NH, 16)).pin_memory()
    else:
        tdt = torch.float16 if dt == "f16" else torch.bfloat16
        gk, gv = W.randn(rng, (N, H, 16, D), tdt), W.randn(rng, (N, H, 16, D), tdt)
        gks = gvs = hks = hvs = None
        hk = torch.zeros((NH, H, 16, D), dtype=tdt).pin_memory()
        hv = torch.zeros_like(hk).pin_memory()
    dk, dv = gk.to(DEV), gv.to(DEV)
    dks = gks.to(DEV) if gks is not None else None
    dvs = gvs.to(DEV) if gvs is not None else None
    out_pairs = np.stack([rng.choice(N, 30, replace=False), rng.choice(NH, 30, replace=False)], 1)
    ops.swap_blocks(hk, hv, dk, dv, torch.from_numpy(out_pairs).to(DEV), hks, hvs, dks, dvs)
    torch.cuda.synchronize()
    ek, ev, eks, evs = o_swap(np.zeros_like(np_exact(hk)), np.zeros_like(np_exact(hv)), np_exact(gk),
                              np_exact(gv), out_pairs, None if hks is None else np.zeros((NH, 16), np.float32),
                              None if hvs is None else np.zeros((NH, 16), np.float32),
                              None if gks is None else gks.numpy(), None if gvs is None else gvs.numpy())
    assert np.array_equal(np_exact(hk), ek) and np.array_equal(np_exact(hv), ev)
    if hks is not None:
        assert np.array_equal(hks.numpy(), eks) and np.array_equal(hvs.numpy(), evs)
    # swap back into other GPU blocks; pairs given in pinned host memory this time
    in_pairs = np.stack([out_pairs[:, 1], rng.choice(N, 30, replace=False)], 1)
    ops.swap_blocks(dk, dv, hk, hv, torch.from_numpy(in_pairs).pin_memory(), dks, dvs, hks, hvs)
    torch.cuda.synchronize()
    fk, fv, fks, fvs = o_swap(np_exact(gk), np_exact(gv), ek, ev, in_pairs,
                              None if gks is None else gks.numpy(), None if gvs is None else gvs.numpy(),
                              eks, evs)
    assert np.array_equal(np_exact(dk), fk) and np.array_equal(np_exact(dv), fv)
    if dks is not None:
        assert np.array_equal(dks.cpu().numpy(), fks) and np.array_equal(dvs.cpu().numpy(), fvs)


def test_preempt_and_resume_keeps_decode_bit_identical():
    w = W.config_llama7b(B=6)
    H, D = w.Hkv, w.D
    gpu = ops.BlockAllocator(w.num_blocks, w.free_order)
    host = ops.BlockAllocator(256)
    ids = list(range(w.B))
    for b in ids:
        gpu.alloc_seq(b, int(w.context_lens[b]))
    kc, vc = w.k_pool.to(DEV), w.v_pool.to(DEV)
    hk = torch.empty((256, H, 16, D), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    cap = -(-int(w.context_lens.max()) // 16)

    def decode():
        tab, lens = gpu.tables(ids, cap)
        out = ops.decode(w.q.to(DEV), kc, vc, torch.from_numpy(tab).to(DEV), torch.from_numpy(lens).to(DEV),
                         int(lens.max()), w.scale, out_dtype=torch.float32)
        torch.cuda.synchronize()
        return out.cpu()

    before = decode()
    victims = [1, 4]
    for s in victims:  # preempt: pages to host, GPU blocks released
        blocks, n = gpu.table(s)
        host.alloc_seq(s, n)
        hblocks, _ = host.table(s)
        pairs = torch.tensor(list(zip(blocks, hblocks)), dtype=torch.int64, device=DEV)
        ops.swap_blocks(hk, hv, kc, vc, pairs)
        torch.cuda.synchronize()
        gpu.free_seq(s)
    filler = 99  # the released blocks are reused (and overwritten) meanwhile
    gpu.alloc_seq(filler, 16 * 40)
    fb, _ = gpu.table(filler)
    kc[torch.tensor(fb, device=DEV)] = 7.0
    vc[torch.tensor(fb, device=DEV)] = -7.0
    gpu.free_seq(filler)
    for s in victims:  # resume: fresh GPU blocks, pages back from host
        hblocks, n = host.table(s)
        gpu.alloc_seq(s, n)
        blocks, _ = gpu.table(s)
        pairs = torch.tensor(list(zip(hblocks, blocks)), dtype=torch.int64, device=DEV)
        ops.swap_blocks(kc, vc, hk, hv, pairs)
        host.free_seq(s)
    after = decode()
    assert torch.equal(before, after)
