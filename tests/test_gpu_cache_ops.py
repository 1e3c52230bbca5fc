"""GPU parity of pa_cache_write and pa_copy_blocks: bit-exact against the
oracle (byte movement and a deterministic quantiser)."""
import numpy as np
import pytest
import torch

from oracle.cache_ops import cache_write as o_write, copy_blocks as o_copy
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import np_exact, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


def _pool(seed, N, H, D, dt):
    rng = W.rng_for(seed)
    return W.randn(rng, (N, H, 16, D), dt), W.randn(rng, (N, H, 16, D), dt)


@pytest.mark.parametrize("kv,inp", [("f16", "f16"), ("bf16", "bf16"), ("f16", "f32"), ("bf16", "f32")])
@pytest.mark.parametrize("H,D,T", [(4, 64, 5), (32, 128, 37), (8, 128, 300)])
def test_write_16bit(kv, inp, H, D, T):
    N = 40
    kc, vc = _pool(1, N, H, D, TD[kv])
    rng = W.rng_for(2)
    k = W.randn(rng, (T, H, D), TD[inp])
    v = W.randn(rng, (T, H, D), TD[inp])
    slots = W.random_slots(3, T, N, n_skip=min(3, T // 4))
    gk, gv = kc.to(DEV), vc.to(DEV)
    ops.cache_write(k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV), gk, gv)
    torch.cuda.synchronize()
    if inp == "f32":  # rounding to the cache dtype is part of the write
        k_in, v_in = np_exact(k.to(TD[kv])), np_exact(v.to(TD[kv]))
    else:
        k_in, v_in = np_exact(k), np_exact(v)
    ek, ev, _, _ = o_write(k_in, v_in, slots, np_exact(kc), np_exact(vc))
    assert np.array_equal(np_exact(gk), ek) and np.array_equal(np_exact(gv), ev)


@pytest.mark.parametrize("inp", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("H,T", [(8, 33), (2, 7)])
@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_write_fp8(inp, H, T, fmt):
    N, D = 24, 128
    rng = W.rng_for(4)
    k = W.randn(rng, (T, H, D), TD[inp]) * 3
    v = W.randn(rng, (T, H, D), TD[inp])
    k[0].zero_()                              # all-zero token -> scale 1, zero codes
    slots = W.random_slots(5, T, N, n_skip=2)
    cdt, lo = (torch.int8, -128) if fmt == "int8" else (torch.uint8, 0)
    kc = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
    vc = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
    ks = torch.rand((N, 16), dtype=torch.float32)
    vs = torch.rand((N, 16), dtype=torch.float32)
    gk, gv, gks, gvs = kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV)
    ops.cache_write(k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV), gk, gv, gks, gvs)
    torch.cuda.synchronize()
    ek, ev, eks, evs = o_write(np_exact(k), np_exact(v), slots, kc.numpy(), vc.numpy(), ks.numpy(), vs.numpy())
    assert np.array_equal(gk.cpu().numpy(), ek) and np.array_equal(gv.cpu().numpy(), ev)
    assert np.array_equal(gks.cpu().numpy(), eks) and np.array_equal(gvs.cpu().numpy(), evs)


def test_write_out_of_range_slot_is_flagged_and_skipped():
    kc, vc = _pool(6, 4, 2, 64, torch.float16)
    k = torch.ones((2, 2, 64), dtype=torch.float16, device=DEV)
    gk, gv = kc.to(DEV), vc.to(DEV)
    ops.cache_write(k, k, torch.tensor([4 * 16 + 3, 5], device=DEV), gk, gv)
    torch.cuda.synchronize()
    assert ops.device_errors(clear=True) & ops.DEVERR_SLOT_RANGE
    ek, _, _, _ = o_write(np.ones((1, 2, 64), np.float16), np.ones((1, 2, 64), np.float16),
                          np.array([5]), np_exact(kc), np_exact(vc))
    assert np.array_equal(np_exact(gk), ek)


@pytest.mark.parametrize("dt", ["f16", "bf16", "fp8", "int8"])
@pytest.mark.parametrize("H,D,n", [(32, 128, 19), (8, 128, 1), (4, 64, 40)])
def test_copy_blocks(dt, H, D, n):
    if dt in ("fp8", "int8") and D != 128:
        pytest.skip("FP8 / INT8 caches are built for head_dim 128")
    N = 100
    if dt in ("fp8", "int8"):
        cdt, lo = (torch.int8, -128) if dt == "int8" else (torch.uint8, 0)
        kc = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
        vc = torch.randint(lo, lo + 255, (N, H, 16, D), dtype=cdt)
        ks, vs = torch.rand((N, 16)), torch.rand((N, 16))
    else:
        kc, vc = _pool(7, N, H, D, TD[dt])
        ks = vs = None
    pairs = W.random_pairs(8, N, n)
    gk, gv = kc.to(DEV), vc.to(DEV)
    gks = ks.to(DEV) if ks is not None else None
    gvs = vs.to(DEV) if vs is not None else None
    ops.copy_blocks(gk, gv, torch.from_numpy(pairs).to(DEV), gks, gvs)
    torch.cuda.synchronize()
    ek, ev, eks, evs = o_copy(np_exact(kc), np_exact(vc), pairs,
                              None if ks is None else ks.numpy(), None if vs is None else vs.numpy())
    assert np.array_equal(np_exact(gk), ek) and np.array_equal(np_exact(gv), ev)
    if ks is not None:
        assert np.array_equal(gks.cpu().numpy(), eks) and np.array_equal(gvs.cpu().numpy(), evs)
