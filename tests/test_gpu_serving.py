"""The whole serving iteration on the GPU against the oracle, step by step:
the native engine (pa_serve_step) turns the C++ scheduler's decisions
(admission, chunked prefill, decode, swap-out, swap-in, drop) into
pa_swap_blocks, pa_decode_append for the decode items and pa_cache_write +
pa_chunked_prefill for the prompt chunks;
the oracle applies the same copies and writes to its own cache mirror and
computes the attention of every new token.  Outputs must agree within the
attention tolerance (plus half an ulp of the 16-bit output) and the device
caches must equal the mirror bit for bit.  The pool is small enough that
requests are preempted both by swap and by drop.  With FP8 / INT8 caches the
mirror holds codes and per-token scales written by the oracle's quantiser,
codes and scales must match bit for bit, and attention is checked on them
within the FP8 / INT8 tolerance."""
import numpy as np
import pytest
import torch

from oracle.attention import paged_prefill
from oracle.cache_ops import cache_write as oracle_cache_write
from oracle.scheduler import Scheduler as OSched
from paged_kv_cache_191_gb300 import ops, workloads as W
from paged_kv_cache_191_gb300.serving import ServingLoop
from tests.gpu_util import TOL, np_exact, half_ulp, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


@pytest.mark.parametrize("dtype,two_phase,kv", [("f16", False, None), ("bf16", False, None), ("f16", True, None),
                                                ("f16", False, "fp8"), ("bf16", True, "int8")])
def test_serving_iterations_match_oracle(dtype, two_phase, kv):
    """two_phase: plan() first, then exactly T rows of q / K / V, then
    launch() -- the order a model feeding the loop follows.  kv: a 1-byte
    cache format (None: the model's 16-bit dtype)."""
    tdt = W.KV_TORCH[dtype]
    nb, hb, Hkv, Hq, D, mb, mt = 12, 6, 2, 8, 128, 4, 48
    q8 = kv is not None
    kvt = {"fp8": torch.uint8, "int8": torch.int8}.get(kv)
    loop = ServingLoop(nb, hb, Hkv, Hq, D, tdt, mb, mt, 256, kv_dtype=kvt)
    ref = OSched(nb, mb, mt, hb)
    rng = W.rng_for(77)
    reqs = []
    for i in range(12):
        while True:
            p, m = int(rng.integers(1, 121)), int(rng.integers(1, 41))
            if -(-(p + m) // 16) <= nb:
                break
        reqs.append((int(rng.integers(0, 25)), 500 + i, p, m))
    cdt = {"fp8": np.uint8, "int8": np.int8}.get(kv, np.float32)
    kc = np.zeros((nb, Hkv, 16, D), cdt)
    vc = np.zeros_like(kc)
    kh = np.zeros((hb, Hkv, 16, D), cdt)
    vh = np.zeros_like(kh)
    ks, vs = np.zeros((nb, 16), np.float32), np.zeros((nb, 16), np.float32)  # per-token scales (1-byte caches)
    khs, vhs = np.zeros((hb, 16), np.float32), np.zeros((hb, 16), np.float32)
    events = {"swap_out": 0, "swap_in": 0, "recomputed": 0, "tokens": 0}
    for it in range(2000):
        for t, rid, p, m in reqs:
            if t == it:
                loop.add(rid, p, m)
                ref.add(rid, p, m)
        if two_phase:
            T_rows = max(loop.plan(), 1)
        else:
            T_rows = mb + mt
        q = W.randn(rng, (T_rows, Hq, D), tdt).cuda()
        kn = W.randn(rng, (T_rows, Hkv, D), tdt).cuda()
        vn = W.randn(rng, (T_rows, Hkv, D), tdt).cuda()
        if two_phase:
            loop.launch(q, kn, vn)
            st = loop.decisions()
        else:
            st = loop.step(q, kn, vn)
        torch.cuda.synchronize()
        r = ref.step()
        # the scheduler decisions are the oracle's
        assert [(i, s, n) for i, s, n in zip(st["ids"], st["starts"], st["lens"])] == \
            [(i, s, len(sl)) for i, _, s, sl in r.items]
        assert list(st["slots"]) == [x for *_, sl in r.items for x in sl]
        assert np.array_equal(st["context_lens"], st["starts"] + st["lens"])
        assert [tuple(x) for x in st["swap_out"]] == r.swap_out
        assert [tuple(x) for x in st["swap_in"]] == r.swap_in
        # the same device work on the mirror, in the same order
        for g, h in r.swap_out:
            kh[h], vh[h], khs[h], vhs[h] = kc[g], vc[g], ks[g], vs[g]
        T = st["T"]
        if T:
            slots = st["slots"]
            if q8:
                kc, vc, ks, vs = oracle_cache_write(np_exact(kn[:T].cpu()), np_exact(vn[:T].cpu()), slots,
                                                    kc, vc, ks, vs)
            else:
                kc[slots // 16, :, slots % 16, :] = np_exact(kn[:T].cpu())
                vc[slots // 16, :, slots % 16, :] = np_exact(vn[:T].cpu())
            qs = np.concatenate([[0], np.cumsum(st["lens"])])
            lens = st["starts"] + st["lens"]
            want = paged_prefill(np_exact(q[:T].cpu()), qs, kc, vc, st["tables"], lens, 1.0 / np.sqrt(D),
                                 k_scale=ks if q8 else None, v_scale=vs if q8 else None)
            got = st["out"].float().cpu().numpy()
            err = np.abs(got - want)
            assert np.all(err <= TOL[kv or dtype] + half_ulp(want, tdt)), (it, float(err.max()))
        for h, g in r.swap_in:
            kc[g], vc[g], ks[g], vs[g] = kh[h], vh[h], khs[h], vhs[h]
        events["swap_out"] += len(r.swap_out)
        events["swap_in"] += len(r.swap_in)
        events["recomputed"] += len(r.recomputed)
        events["tokens"] += T
        if ref.idle() and it > 25:
            break
    assert loop.idle()
    torch.cuda.synchronize()
    if q8:
        assert np.array_equal(loop.k_cache.cpu().numpy(), kc) and np.array_equal(loop.v_cache.cpu().numpy(), vc)
        assert np.array_equal(loop.k_scale.cpu().numpy(), ks) and np.array_equal(loop.v_scale.cpu().numpy(), vs)
    else:
        assert np.array_equal(np_exact(loop.k_cache.cpu()), kc) and np.array_equal(np_exact(loop.v_cache.cpu()), vc)
    assert events["swap_out"] and events["swap_in"] and events["recomputed"], events
