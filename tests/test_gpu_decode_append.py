"""pa_decode_append (cache write fused into decode) against the two separate
calls: outputs, cache contents and FP8 / INT8 scales must be bit-identical,
and both within tolerance of the oracle."""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode
from oracle.cache_ops import cache_write as o_write
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, assert_close, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


def last_slots(w):
    """Slot of each sequence's last token through its table (-1 for L = 0)."""
    L = w.context_lens.astype(np.int64)
    blk = w.block_tables[np.arange(w.B), np.maximum(L - 1, 0) // 16].astype(np.int64)
    return np.where(L > 0, blk * 16 + (L - 1) % 16, -1)


def fp8_caches(w):
    N, H, _, D = w.k_pool.shape
    kin = w.k_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    vin = w.v_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    kc = torch.empty((N, H, 16, D), dtype=torch.int8 if w.kv_dtype == "int8" else torch.uint8, device=DEV)
    vc = torch.empty_like(kc)
    ks = torch.empty((N, 16), dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    ops.cache_write(kin, vin, torch.arange(N * 16, device=DEV), kc, vc, ks, vs)
    return kc, vc, ks, vs


@pytest.mark.parametrize("Hq,Hkv,kv,inp,split", [
    (8, 8, "f16", "f16", 0), (32, 4, "bf16", "bf16", 64), (16, 2, "f16", "f32", 16),
    (16, 4, "fp8", "f16", 0), (8, 2, "fp8", "f32", 64), (8, 8, "fp8", "bf16", 0),
    (16, 4, "int8", "f16", 0), (8, 2, "int8", "f32", 64), (8, 8, "int8", "bf16", 0),
])
def test_fused_equals_write_then_decode(Hq, Hkv, kv, inp, split):
    w = W.random_small(71 + Hq + Hkv, B=7, Hq=Hq, Hkv=Hkv, D=128, kv_dtype=kv, max_len=600, min_len=1)
    q = w.q.to(torch.bfloat16) if kv == "bf16" else w.q
    slots = last_slots(w)
    slots[3] = -1                      # a padding row: nothing stored
    rng = W.rng_for(3)
    k_new = W.randn(rng, (w.B, Hkv, 128), TD[inp]).to(DEV)
    v_new = W.randn(rng, (w.B, Hkv, 128), TD[inp]).to(DEV)
    sl = torch.from_numpy(slots).to(DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    ml = int(w.context_lens.max())
    results = []
    for fused in (False, True):
        if kv in ("fp8", "int8"):
            kc, vc, ks, vs = fp8_caches(w)
        else:
            kc, vc, ks, vs = w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
        if fused:
            out = ops.decode_append(k_new, v_new, sl, q.to(DEV), kc, vc, bt, cl, ml, w.scale,
                                    out_dtype=torch.float32, k_scale=ks, v_scale=vs, split_tokens=split)
        else:
            ops.cache_write(k_new, v_new, sl, kc, vc, ks, vs)
            out = ops.decode(q.to(DEV), kc, vc, bt, cl, ml, w.scale, out_dtype=torch.float32,
                             k_scale=ks, v_scale=vs, split_tokens=split)
        torch.cuda.synchronize()
        results.append([t.cpu() for t in (out, kc, vc) + ((ks, vs) if ks is not None else ())])
    for a, b in zip(*results):
        assert torch.equal(a, b), "fused and separate paths differ"
    if kv not in ("fp8", "int8"):
        kin = np_exact(k_new.cpu().to(TD[kv])) if inp == "f32" else np_exact(k_new.cpu())
        vin = np_exact(v_new.cpu().to(TD[kv])) if inp == "f32" else np_exact(v_new.cpu())
        okc, ovc, _, _ = o_write(kin, vin, slots, np_exact(w.k_pool), np_exact(w.v_pool))
        assert np.array_equal(np_exact(results[1][1]), okc) and np.array_equal(np_exact(results[1][2]), ovc)
        ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
        assert_close(results[1][0].numpy(), ref, TOL[kv], "fused vs oracle")


@pytest.mark.parametrize("rep", range(6))
@pytest.mark.parametrize("Hkv", [8, 2])
@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_fused_fp8_scales_are_race_free(rep, Hkv, fmt):
    """Every kv head of a token reads the token's fresh scale: repeated runs
    with many heads per sequence (the scale row is shared by all of them)."""
    test_fused_equals_write_then_decode(8 * (Hkv // 2) if Hkv > 2 else 8, Hkv, fmt, "bf16", 0)


@pytest.mark.parametrize("kv", ["f16", "fp8"])
def test_decode_session_equals_decode_append(kv):
    """DecodeSession (one staging copy, one fused launch, one output copy per
    step) gives the same output and cache as ops.decode_append, step after
    step while the ring of host buffers rotates."""
    from paged_kv_cache_191_gb300.session import DecodeSession
    w = W.random_small(123, B=6, Hq=8, Hkv=2, D=128, kv_dtype=kv, max_len=600, min_len=1)
    ml, mb = int(w.context_lens.max()), w.block_tables.shape[1]
    if kv == "fp8":
        kc, vc, ks, vs = fp8_caches(w)
        kc2, vc2, ks2, vs2 = fp8_caches(w)
    else:
        kc, vc, ks, vs = w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
        kc2, vc2, ks2, vs2 = w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
    sess = DecodeSession(kc, vc, w.B, w.Hq, mb, ml, w.scale, torch.float16, k_scale=ks, v_scale=vs,
                         out_dtype=torch.float32, items=False)
    rng = W.rng_for(9)
    for step in range(3):
        k_new = W.randn(rng, (w.B, w.Hkv, 128), torch.float16)
        v_new = W.randn(rng, (w.B, w.Hkv, 128), torch.float16)
        slots_p, lens_p, tab_p = sess.meta_ptrs()
        np.ctypeslib.as_array(slots_p, (w.B,))[:] = last_slots(w)
        np.ctypeslib.as_array(lens_p, (w.B,))[:] = w.context_lens
        np.ctypeslib.as_array(tab_p, (w.B, mb))[:] = w.block_tables
        q, k, v = sess.inputs()
        q.copy_(w.q)
        k.copy_(k_new)
        v.copy_(v_new)
        got = sess.step().clone()
        want = ops.decode_append(k_new.to(DEV), v_new.to(DEV), torch.from_numpy(last_slots(w)).to(DEV),
                                 w.q.to(DEV), kc2, vc2, torch.from_numpy(w.block_tables).to(DEV),
                                 torch.from_numpy(w.context_lens).to(DEV), ml, w.scale, out_dtype=torch.float32,
                                 k_scale=ks2, v_scale=vs2)
        torch.cuda.synchronize()
        assert torch.equal(got, want.cpu()), step
        assert torch.equal(kc.cpu(), kc2.cpu()) and torch.equal(vc.cpu(), vc2.cpu()), step


@pytest.mark.parametrize("kv,mode", [("f16", True), ("f16", "auto"), ("fp8", "auto"), ("bf16", "auto")])
def test_decode_session_items(kv, mode):
    """DecodeSession in items mode over a batch with log-uniform lengths
    (most cells of the fixed grid empty, so "auto" lists too): the session
    lists the live partitions on the host and runs
    pa_decode_append_segments.  Output within 5e-4 of ops.decode_append and
    within tolerance of the oracle, caches and scales bit-identical, step
    after step.  A uniform batch under "auto" stays on the fixed grid and
    matches ops.decode_append bit for bit."""
    from paged_kv_cache_191_gb300.session import DecodeSession
    rng = np.random.default_rng(31)
    lens = np.exp(rng.uniform(np.log(8), np.log(1500), 24)).astype(np.int32)
    w = W.make_decode("skewed", 44, 24, 16, 4, 128, kv, lens, pool_factor=1.3)
    ml, mb = int(w.context_lens.max()), w.block_tables.shape[1]
    dt = torch.bfloat16 if kv == "bf16" else torch.float16
    if kv == "fp8":
        kc, vc, ks, vs = fp8_caches(w)
        kc2, vc2, ks2, vs2 = fp8_caches(w)
    else:
        kc, vc, ks, vs = w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
        kc2, vc2, ks2, vs2 = w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
    assert ops.decode_items_plan(w.context_lens, w.Hq, ml, kc)[0]
    sess = DecodeSession(kc, vc, w.B, w.Hq, mb, ml, w.scale, dt, k_scale=ks, v_scale=vs,
                         out_dtype=torch.float32, items=mode)
    rng = W.rng_for(10)
    for step in range(3):
        k_new = W.randn(rng, (w.B, w.Hkv, 128), dt)
        v_new = W.randn(rng, (w.B, w.Hkv, 128), dt)
        slots_p, lens_p, tab_p = sess.meta_ptrs()
        np.ctypeslib.as_array(slots_p, (w.B,))[:] = last_slots(w)
        np.ctypeslib.as_array(lens_p, (w.B,))[:] = w.context_lens
        np.ctypeslib.as_array(tab_p, (w.B, mb))[:] = w.block_tables
        q, k, v = sess.inputs()
        q.copy_(w.q)
        k.copy_(k_new)
        v.copy_(v_new)
        got = sess.step().clone().numpy()
        assert sess.last_items and sess.last_copy_bytes == sess.nbytes + 16 * sess.last_items
        want = ops.decode_append(k_new.to(DEV), v_new.to(DEV), torch.from_numpy(last_slots(w)).to(DEV),
                                 w.q.to(DEV), kc2, vc2, torch.from_numpy(w.block_tables).to(DEV),
                                 torch.from_numpy(w.context_lens).to(DEV), ml, w.scale, out_dtype=torch.float32,
                                 k_scale=ks2, v_scale=vs2)
        torch.cuda.synchronize()
        assert np.abs(got - want.cpu().numpy()).max() <= 5e-4, step
        assert torch.equal(kc.cpu(), kc2.cpu()) and torch.equal(vc.cpu(), vc2.cpu()), step
        if kv == "fp8":
            assert torch.equal(ks.cpu(), ks2.cpu()) and torch.equal(vs.cpu(), vs2.cpu()), step
            ref = paged_decode(np_exact(w.q), kc.cpu().numpy(), vc.cpu().numpy(), w.block_tables, w.context_lens,
                               w.scale, k_scale=ks.cpu().numpy(), v_scale=vs.cpu().numpy())
        else:
            ref = paged_decode(np_exact(w.q), np_exact(kc.cpu()), np_exact(vc.cpu()), w.block_tables,
                               w.context_lens, w.scale)
        assert_close(got, ref, TOL[kv], f"session items {kv} step {step}")
    # uniform lengths: "auto" keeps the fixed grid
    wu = W.make_decode("uniform", 45, 8, 16, 4, 128, "f16", np.full(8, 700, np.int32), pool_factor=1.3)
    mlu, mbu = 700, wu.block_tables.shape[1]
    kcu, vcu = wu.k_pool.to(DEV), wu.v_pool.to(DEV)
    kcu2, vcu2 = wu.k_pool.to(DEV), wu.v_pool.to(DEV)
    assert not ops.decode_items_plan(wu.context_lens, wu.Hq, mlu, kcu)[0]
    sess = DecodeSession(kcu, vcu, wu.B, wu.Hq, mbu, mlu, wu.scale, torch.float16, out_dtype=torch.float32)
    slots_p, lens_p, tab_p = sess.meta_ptrs()
    np.ctypeslib.as_array(slots_p, (wu.B,))[:] = last_slots(wu)
    np.ctypeslib.as_array(lens_p, (wu.B,))[:] = wu.context_lens
    np.ctypeslib.as_array(tab_p, (wu.B, mbu))[:] = wu.block_tables
    q, k, v = sess.inputs()
    q.copy_(wu.q)
    k.copy_(wu.new_k)
    v.copy_(wu.new_v)
    got = sess.step().clone()
    assert sess.last_items is None and sess.last_copy_bytes == sess.nbytes
    want = ops.decode_append(wu.new_k.to(DEV), wu.new_v.to(DEV), torch.from_numpy(last_slots(wu)).to(DEV),
                             wu.q.to(DEV), kcu2, vcu2, torch.from_numpy(wu.block_tables).to(DEV),
                             torch.from_numpy(wu.context_lens).to(DEV), mlu, wu.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(got, want.cpu())
