"""The C ABI: every declared entry point is exported, and host-side
validation rejects bad calls before anything is launched (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from paged_kv_cache_191_gb300 import ops
from tests.libfixture import palib  # noqa: F401

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(palib):
    names = declared_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(palib, n), f"{n} not exported by libpagedkv.so"
    assert set(names) == set(ops.SIGNATURES), "binding and header disagree"


def test_version(palib):
    assert palib.pa_version() == 100


def _desc(**kw):
    d = dict(num_blocks=8, num_kv_heads=2, head_dim=128, block_size=16, kv_dtype=ops.F16)
    d.update(kw)
    return ops.CacheDesc(**d)


FAKE = 0x10000  # 16-byte aligned dummy address; never dereferenced on a rejected call


def _decode(desc, **kw):
    a = dict(q=FAKE, q_dtype=ops.F16, k=FAKE, v=FAKE, ks=None, vs=None, bt=FAKE, maxb=4, cl=FAKE,
             maxl=64, B=2, Hq=4, scale=0.1, out=FAKE, odt=ops.F16, ws=None, wsb=0, split=0)
    a.update(kw)
    lib = ops.lib()
    return lib.pa_decode(a["q"], a["q_dtype"], a["k"], a["v"], a["ks"], a["vs"], a["bt"], a["maxb"],
                         a["cl"], a["maxl"], a["B"], a["Hq"], a["scale"], a["out"], a["odt"],
                         C.byref(desc), a["ws"], a["wsb"], a["split"], None)


@pytest.mark.parametrize("desc_kw,call_kw,status", [
    ({"block_size": 32}, {}, ops.PA_ERR_UNSUPPORTED),
    ({"head_dim": 96}, {}, ops.PA_ERR_UNSUPPORTED),
    ({"kv_dtype": 7}, {}, ops.PA_ERR_INVALID),
    ({"kv_dtype": ops.FP8_E4M3, "head_dim": 64}, {}, ops.PA_ERR_UNSUPPORTED),
    ({}, {"Hq": 3}, ops.PA_ERR_INVALID),                 # not a multiple of Hkv
    ({}, {"Hq": 32}, ops.PA_ERR_UNSUPPORTED),            # group of 16 > 8
    ({}, {"q": None}, ops.PA_ERR_INVALID),
    ({}, {"out": FAKE + 4}, ops.PA_ERR_INVALID),         # misaligned
    ({}, {"q_dtype": ops.BF16}, ops.PA_ERR_INVALID),     # q dtype != cache dtype
    ({}, {"odt": ops.BF16}, ops.PA_ERR_INVALID),
    ({}, {"scale": float("nan")}, ops.PA_ERR_INVALID),
    ({}, {"maxl": 4096, "split": 256}, ops.PA_ERR_INVALID),  # needs a workspace
    ({}, {"maxl": 4096, "split": 24}, ops.PA_ERR_INVALID),   # not a multiple of 16
    ({"kv_dtype": ops.FP8_E4M3}, {}, ops.PA_ERR_INVALID),    # FP8 without scales
    ({}, {"ks": FAKE}, ops.PA_ERR_INVALID),                  # scales on a 16-bit cache
])
def test_decode_rejects_bad_arguments(palib, desc_kw, call_kw, status):
    assert _decode(_desc(**desc_kw), **call_kw) == status
    assert palib.pa_last_error()


def test_decode_workspace_size(palib):
    """One partition needs no workspace.  A split needs the partials (o, m, l
    per sequence, query head and partition) and, when it has at most 8
    partitions, one 8-byte arrival counter per (sequence, kv head) after them
    for the in-kernel merge."""
    d = _desc()
    B, Hq, Hkv = 4, 4, 2
    assert palib.pa_decode_workspace_size(B, Hq, 256, C.byref(d), 256) == 0
    ws = palib.pa_decode_workspace_size(B, Hq, 1000, C.byref(d), 256)
    # 4 partitions of 256 tokens: o [B*Hq*4*128] f32 + m, l [B*Hq*4] f32, then the counters
    partials = (B * Hq * 4 * (128 + 2) * 4 + 255) // 256 * 256
    assert ws == partials + (B * Hkv * 8 + 255) // 256 * 256
    # 16 partitions: merged by the merge kernel, no counters
    ws16 = palib.pa_decode_workspace_size(B, Hq, 4000, C.byref(d), 256)
    assert ws16 == (B * Hq * 16 * (128 + 2) * 4 + 255) // 256 * 256


def test_cache_write_and_copy_reject_bad_arguments(palib):
    d = _desc()
    lib = ops.lib()
    assert lib.pa_cache_write(FAKE, FAKE, ops.BF16, FAKE, 3, FAKE, FAKE, None, None, C.byref(d), None) == ops.PA_ERR_INVALID
    assert lib.pa_cache_write(FAKE, None, ops.F16, FAKE, 3, FAKE, FAKE, None, None, C.byref(d), None) == ops.PA_ERR_INVALID
    assert lib.pa_cache_write(FAKE, FAKE, ops.F16, FAKE, 0, FAKE, FAKE, None, None, C.byref(d), None) == ops.PA_OK
    assert lib.pa_copy_blocks(FAKE, FAKE, None, None, FAKE, -1, C.byref(d), None) == ops.PA_ERR_INVALID
    assert lib.pa_copy_blocks(FAKE, FAKE, None, None, FAKE, 0, C.byref(d), None) == ops.PA_OK
    d8 = _desc(kv_dtype=ops.FP8_E4M3)
    assert lib.pa_copy_blocks(FAKE, FAKE, None, None, FAKE, 2, C.byref(d8), None) == ops.PA_ERR_INVALID


def _grouped(desc, **kw):
    a = dict(kn=FAKE, vn=FAKE, ndt=ops.F16, slots=FAKE, q=FAKE, q_dtype=ops.F16, k=FAKE, v=FAKE, ks=None, vs=None,
             bt=FAKE, maxb=8, cl=FAKE, maxl=128, B=8, Hq=4, scale=0.1, gs=FAKE, pre=FAKE, ng=2, mg=4, mp=4,
             out=FAKE, odt=ops.F16, ws=None, wsb=0, split=0)
    a.update(kw)
    return ops.lib().pa_decode_append_grouped(
        a["kn"], a["vn"], a["ndt"], a["slots"], a["q"], a["q_dtype"], a["k"], a["v"], a["ks"], a["vs"], a["bt"],
        a["maxb"], a["cl"], a["maxl"], a["B"], a["Hq"], a["scale"], a["gs"], a["pre"], a["ng"], a["mg"], a["mp"],
        a["out"], a["odt"], C.byref(desc), a["ws"], a["wsb"], a["split"], None)


@pytest.mark.parametrize("call_kw,status", [
    ({"mg": 5}, ops.PA_ERR_UNSUPPORTED),           # 5 members x G = 2 -> 10 query columns > 8
    ({"ng": 0}, ops.PA_ERR_INVALID),
    ({"ng": 9}, ops.PA_ERR_INVALID),               # more groups than sequences
    ({"mp": -1}, ops.PA_ERR_INVALID),
    ({"gs": None}, ops.PA_ERR_INVALID),
    ({"pre": FAKE + 2}, ops.PA_ERR_INVALID),       # misaligned
    ({"slots": None}, ops.PA_ERR_INVALID),
    ({}, ops.PA_ERR_INVALID),                      # a grouped call always needs its workspace
])
def test_grouped_decode_rejects_bad_arguments(palib, call_kw, status):
    assert _grouped(_desc(), **call_kw) == status
    assert palib.pa_last_error()


def test_grouped_workspace_size(palib):
    d = _desc()  # Hkv = 2; Hq = 4 -> G = 2
    # 128-token contexts (8 blocks), prefix of 4 blocks, 512-token partitions:
    # one prefix partition + one tail partition per member
    ws = palib.pa_decode_grouped_workspace_size(8, 4, 128, 2, 4, 4, C.byref(d), 0)
    assert ws >= 8 * 4 * 2 * (128 + 2) * 4 and ws % 256 == 0
    assert palib.pa_decode_grouped_workspace_size(8, 4, 128, 2, 5, 4, C.byref(d), 0) == 0  # 10 columns
    assert palib.pa_decode_grouped_workspace_size(8, 4, 128, 0, 4, 4, C.byref(d), 0) == 0


def test_chunked_prefill_scale_rules(palib):
    """1-byte caches need 16-byte aligned scales and a 16-bit q; 16-bit caches take none."""
    lib = ops.lib()

    def call(desc, q_dtype, ks, vs):
        return lib.pa_chunked_prefill(FAKE, q_dtype, FAKE, 4, 4, FAKE, FAKE, ks, vs, FAKE, 4, FAKE, 64, 1, 4, 0.1,
                                      FAKE, ops.F32, C.byref(desc), None, 0, 0, None)
    d8 = _desc(kv_dtype=ops.FP8_E4M3)
    assert call(d8, ops.F16, None, None) == ops.PA_ERR_INVALID
    assert call(d8, ops.F16, FAKE + 4, FAKE) == ops.PA_ERR_INVALID
    assert call(d8, ops.FP8_E4M3, FAKE, FAKE) == ops.PA_ERR_INVALID
    assert call(_desc(), ops.F16, FAKE, FAKE) == ops.PA_ERR_INVALID
    assert call(_desc(), ops.BF16, None, None) == ops.PA_ERR_INVALID


def test_plan_info_counts_the_kernels_a_call_launches(palib):
    """pa_decode_plan_info: one partition -> 1 kernel; up to 8 partitions ->
    1 (the decode kernel merges them); more -> 2 (a merge kernel follows).
    pa_chunked_prefill_plan_info adds the decode kernel's launches for the
    one-token sequences, and a call whose longest query is one token
    launches only those."""
    d = _desc()
    assert ops.decode_plan_info(4, 4, 256, _torch_like(d), 256) == (1, 16, 1)
    assert ops.decode_plan_info(4, 4, 2048, _torch_like(d), 256) == (8, 16, 1)
    assert ops.decode_plan_info(4, 4, 4096, _torch_like(d), 256) == (16, 16, 2)
    d8 = _desc(kv_dtype=ops.FP8_E4M3)
    dec8 = ops.decode_plan_info(8, 4, 300, _torch_like(d8))[2]
    # 40 tokens x 2 heads per kv head = 80 rows: the tcgen05 kernel (128-row tiles)
    tc, parts, bpp, k = ops.chunked_prefill_plan_info(70, 8, 4, 40, 300, _torch_like(d8), 0)
    assert tc == 1 and k == 1 + (1 if parts > 1 else 0) + dec8
    # 30 x 2 = 60 rows: the 64-row kernel
    tc, parts, bpp, k = ops.chunked_prefill_plan_info(60, 8, 4, 30, 300, _torch_like(d8), 0)
    assert tc == 0 and k == 1 + (1 if parts > 1 else 0) + dec8
    assert ops.chunked_prefill_plan_info(8, 8, 4, 1, 300, _torch_like(d8), 0)[3] == \
        ops.decode_plan_info(8, 4, 300, _torch_like(d8))[2]
    # 16-bit caches alike: the decode kernel takes the one-token sequences
    tc, parts, bpp, k = ops.chunked_prefill_plan_info(70, 8, 4, 40, 300, _torch_like(d), 0)
    assert k == 1 + (1 if parts > 1 else 0) + ops.decode_plan_info(8, 4, 300, _torch_like(d))[2]


def test_short_queries_go_to_the_decode_kernel(palib):
    """A 16-bit cache with at most 8 query tokens per sequence and 32 rows per
    kv head: the decode kernel serves the whole call, one grid column per
    query token, so the plan is the decode plan for B x max_q_len rows.
    More rows, or a 1-byte cache, keep the multi-token kernels.  The
    workspace size covers every call up to its bounds, short ones included."""
    dg = _desc(num_kv_heads=8, kv_dtype=ops.BF16)
    for mq in (1, 2, 4):
        tc, parts, bpp, k = ops.chunked_prefill_plan_info(64 * mq, 64, 64, mq, 4096, _torch_like(dg), 0)
        assert (tc, parts, bpp, k) == (0, *ops.decode_plan_info(64 * mq, 64, 4096, _torch_like(dg)))
    # 5 tokens x 8 heads = 40 rows: the 64-row kernel (+ its merge when split),
    # and the decode kernel for one-token sequences
    tc, parts, bpp, k = ops.chunked_prefill_plan_info(64 * 5, 64, 64, 5, 4096, _torch_like(dg), 0)
    assert tc == 0 and k == 1 + (parts > 1) + ops.decode_plan_info(64, 64, 4096, _torch_like(dg))[2]
    # G = 1: up to 8 tokens take the decode route
    d1 = _desc(num_kv_heads=32, kv_dtype=ops.F16)
    assert ops.chunked_prefill_plan_info(8 * 8, 8, 32, 8, 2048, _torch_like(d1), 0)[1:] == \
        ops.decode_plan_info(8 * 8, 32, 2048, _torch_like(d1))
    # 1-byte codes, 2 tokens: the multi-token kernel (+ the decode kernel for one-token sequences)
    d8 = _desc(num_kv_heads=8, kv_dtype=ops.FP8_E4M3)
    tc, parts, bpp, k = ops.chunked_prefill_plan_info(64 * 2, 64, 64, 2, 4096, _torch_like(d8), 0)
    assert k == 1 + (parts > 1) + ops.decode_plan_info(64, 64, 4096, _torch_like(d8))[2]
    # sizes: a bound of 512 query tokens covers a 2-token call of the same batch
    lib = ops.lib()
    size = lambda mq: lib.pa_chunked_prefill_workspace_size(2076, 32, 32, mq, 2048, C.byref(d1), 0)
    assert size(512) >= size(2) > 0


def _torch_like(desc):
    """A CPU tensor with the cache shape and dtype a desc describes (the plan
    calls read only its shape and dtype)."""
    import torch
    dt = {ops.F16: torch.float16, ops.BF16: torch.bfloat16, ops.FP8_E4M3: torch.uint8, ops.INT8: torch.int8}
    return torch.empty((desc.num_blocks, desc.num_kv_heads, desc.block_size, desc.head_dim), dtype=dt[desc.kv_dtype])


def test_items_plan_follows_the_live_cell_count(palib):
    """pa_decode_items_plan: the item list when fewer than half of the fixed
    grid's (sequence, partition) cells hold blocks, the split has more than
    one partition and G <= 8; blocks_per_item is the plan's partition length
    and max_items_per_seq its partition count."""
    import numpy as np
    dg = _desc(num_kv_heads=8, kv_dtype=ops.BF16)
    rng = np.random.default_rng(5)
    skewed = np.exp(rng.uniform(np.log(16), np.log(4096), 64)).astype(np.int32)   # log-uniform lengths
    uniform = rng.integers(1, 2049, 32).astype(np.int32)
    assert ops.decode_items_plan(skewed, 64, 4096, _torch_like(dg)) == (True, 32, 8)
    d1 = _desc(num_kv_heads=32)
    assert ops.decode_items_plan(uniform, 32, 2048, _torch_like(d1)) == (False, 32, 4)
    # the rule, checked against its definition on random batches
    for trial in range(40):
        B = int(rng.integers(1, 80))
        maxl = int(rng.integers(1, 9000))
        lens = (rng.integers(0, maxl + 1, B) if trial % 2 else
                np.minimum(maxl, np.exp(rng.uniform(0, np.log(maxl + 1), B)))).astype(np.int32)
        for Hq, d in ((64, dg), (32, d1)):
            parts, bpp, _ = ops.decode_plan_info(B, Hq, maxl, _torch_like(d))
            live = int(((lens + 15) // 16 + bpp - 1).__floordiv__(bpp).sum())
            want = parts > 1 and 2 * live < B * parts
            assert ops.decode_items_plan(lens, Hq, maxl, _torch_like(d)) == (want, bpp, max(1, parts))
    # G = 16 never lists: a member's query heads fill one MMA's 8 columns
    d16 = _desc(num_kv_heads=4, kv_dtype=ops.BF16)
    assert ops.decode_items_plan(skewed, 64, 4096, _torch_like(d16))[0] is False
    # one partition (a 256-token split of 256-token contexts): nothing to skip
    assert ops.decode_items_plan(np.full(8, 16, np.int32), 64, 256, _torch_like(dg), 256) == (False, 16, 1)
    # a length past max_context_len, and a null pointer
    with pytest.raises(RuntimeError):
        ops.decode_items_plan(np.array([5000], np.int32), 64, 4096, _torch_like(dg))
    use = C.c_int32()
    assert palib.pa_decode_items_plan(None, 1, 64, 4096, C.byref(dg), 0, C.byref(use), None, None) == \
        ops.PA_ERR_INVALID
