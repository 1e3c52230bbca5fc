"""pa_decode_append_grouped (shared-prefix groups read once per group)
against the oracle and against the ungrouped pa_decode_append.

Groups are built the way fork builds them: every member of a group holds the
same block ids for the first P blocks of its table (a shared prompt), then
private tail blocks.  The fused write of each member's new token must leave
the same cache as the oracle's cache write; outputs must match the oracle
within the attention tolerance and the ungrouped call within 5e-4 (the
partitions differ, so the 16-bit rounding of the softmax weights, taken
against each partition's running max, differs).  Shapes cover G = 1, 2, 4, 8, partition sizes that
cut the prefix into several partitions, groups of one, an empty member, a
claimed prefix longer than the members' contexts allow, and the error flags
for mismatched tables and bad group bounds."""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode
from oracle.cache_ops import cache_write as o_write
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, assert_close, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0


def grouped_case(seed, sizes, prefix, Hq, Hkv, kv, tail_max=60, zero=(), D=128):
    """Lengths 16 * P_k + tail (tail in [1, tail_max]); members of group k
    share their first P_k table entries with the group's first member."""
    rng = W.rng_for(seed)
    lens = []
    for k, n in enumerate(sizes):
        for _ in range(n):
            lens.append(16 * prefix[k] + int(rng.integers(1, tail_max + 1)))
    for b in zero:
        lens[b] = 0
    w = W.make_decode(f"grouped{seed}", seed + 5, len(lens), Hq, Hkv, D, kv, lens, pool_factor=1.3)
    start = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    tables = w.block_tables.copy()
    for k in range(len(sizes)):
        for b in range(start[k] + 1, start[k + 1]):
            if lens[b] > 0 and lens[start[k]] > 0:
                tables[b, :prefix[k]] = tables[start[k], :prefix[k]]
    w.block_tables = tables
    return w, start


def last_slots(w):
    L = w.context_lens.astype(np.int64)
    blk = w.block_tables[np.arange(w.B), np.maximum(L - 1, 0) // 16].astype(np.int64)
    return np.where(L > 0, blk * 16 + (L - 1) % 16, -1)


def caches(w):
    if w.kv_dtype not in ("fp8", "int8"):
        return w.k_pool.to(DEV), w.v_pool.to(DEV), None, None
    N, H, _, D = w.k_pool.shape
    kin = w.k_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    vin = w.v_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    kc = torch.empty((N, H, 16, D), dtype=torch.int8 if w.kv_dtype == "int8" else torch.uint8, device=DEV)
    vc = torch.empty_like(kc)
    ks = torch.empty((N, 16), dtype=torch.float32, device=DEV)
    vs = torch.empty_like(ks)
    ops.cache_write(kin, vin, torch.arange(N * 16, device=DEV), kc, vc, ks, vs)
    return kc, vc, ks, vs


def run(w, start, claimed, split=0, grouped=True, max_size=None):
    rng = W.rng_for(17)
    q = w.q.to(torch.bfloat16) if w.kv_dtype == "bf16" else w.q
    tdt = q.dtype
    k_new = W.randn(rng, (w.B, w.Hkv, w.D), tdt).to(DEV)
    v_new = W.randn(rng, (w.B, w.Hkv, w.D), tdt).to(DEV)
    sl = torch.from_numpy(last_slots(w)).to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables, dtype=np.int32)).to(DEV)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens, dtype=np.int32)).to(DEV)
    ml = max(int(w.context_lens.max()), 1)
    kc, vc, ks, vs = caches(w)
    if grouped:
        gs = torch.from_numpy(start).to(DEV)
        pre = torch.from_numpy(np.asarray(claimed, dtype=np.int32)).to(DEV)
        size = max_size or int(np.diff(start).max())
        out = ops.decode_append_grouped(k_new, v_new, sl, q.to(DEV), kc, vc, bt, cl, ml, w.scale, gs, pre, size,
                                        int(max(claimed)), out_dtype=torch.float32, k_scale=ks, v_scale=vs,
                                        split_tokens=split)
    else:
        out = ops.decode_append(k_new, v_new, sl, q.to(DEV), kc, vc, bt, cl, ml, w.scale, out_dtype=torch.float32,
                                k_scale=ks, v_scale=vs, split_tokens=split)
    torch.cuda.synchronize()
    return out.cpu().numpy(), [t.cpu() if t is not None else None for t in (kc, vc, ks, vs)], (k_new, v_new, q)


CASES = [  # Hq, Hkv, kv, group sizes, shared prefix blocks (head_dim 128; last case 64)
    (8, 8, "f16", [4, 1, 3], [5, 0, 3]),
    (16, 8, "f16", [4, 2, 1, 3], [6, 2, 0, 4]),
    (16, 8, "bf16", [3, 4], [9, 1]),
    (8, 2, "f16", [2, 2, 1], [7, 3, 2]),
    (32, 4, "bf16", [1, 1, 1], [4, 2, 0]),
    (8, 2, "fp8", [2, 1, 2], [6, 0, 3]),
    (16, 8, "int8", [4, 3], [5, 2]),
    (4, 4, "bf16", [3, 2, 4], [4, 6, 1]),
]


@pytest.mark.parametrize("Hq,Hkv,kv,sizes,prefix", CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("split", [0, 32])
def test_grouped_matches_oracle_and_ungrouped(Hq, Hkv, kv, sizes, prefix, split):
    D = 64 if (Hq, Hkv) == (4, 4) else 128
    w, start = grouped_case(50 + Hq + Hkv + len(sizes), sizes, prefix, Hq, Hkv, kv, D=D)
    got, dev_caches, (k_new, v_new, q) = run(w, start, prefix, split)
    plain, plain_caches, _ = run(w, start, prefix, split, grouped=False)
    for a, b in zip(dev_caches, plain_caches):  # the fused writes are the same
        assert a is None or torch.equal(a, b)
    assert np.abs(got - plain).max() <= 5e-4, float(np.abs(got - plain).max())
    slots = last_slots(w)
    kin, vin = np_exact(k_new.cpu()), np_exact(v_new.cpu())
    if kv in ("fp8", "int8"):
        kc, vc, ks, vs = (t.numpy() for t in dev_caches)
        ref = paged_decode(np_exact(q), kc, vc, w.block_tables, w.context_lens, w.scale, k_scale=ks, v_scale=vs)
    else:
        okc, ovc, _, _ = o_write(kin, vin, slots, np_exact(w.k_pool), np_exact(w.v_pool))
        assert np.array_equal(np_exact(dev_caches[0]), okc) and np.array_equal(np_exact(dev_caches[1]), ovc)
        ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL[kv], f"grouped {sizes} {prefix}")


def test_claimed_prefix_is_clamped_and_empty_member():
    """A claimed prefix of 100 blocks is cut to the blocks before every
    member's last token; a group with an empty member shares nothing and the
    empty member gets zero rows."""
    w, start = grouped_case(91, [3, 3], [4, 2], 8, 8, "f16", tail_max=15, zero=(4,))
    got, dev_caches, (k_new, v_new, q) = run(w, start, [100, 100])
    slots = last_slots(w)
    okc, ovc, _, _ = o_write(np_exact(k_new.cpu()), np_exact(v_new.cpu()), slots, np_exact(w.k_pool),
                             np_exact(w.v_pool))
    ref = paged_decode(np_exact(q), okc, ovc, w.block_tables, w.context_lens, w.scale)
    assert_close(got, ref, TOL["f16"], "clamped prefix")
    assert np.all(got[4] == 0.0)


def test_mismatched_tables_and_bad_groups_are_flagged():
    w, start = grouped_case(93, [3, 2], [4, 2], 8, 8, "f16")
    w.block_tables[1, 1] = w.block_tables[1, 5]  # member 1 no longer shares block 1
    run(w, start, [4, 2])
    assert ops.device_errors(clear=True) & ops.DEVERR_GROUP
    w, start = grouped_case(94, [3, 2], [4, 2], 8, 8, "f16")
    run(w, start, [4, 2], max_size=2)  # a group of 3 above the stated bound: skipped
    assert ops.device_errors(clear=True) & ops.DEVERR_GROUP


# ---- the shared-prefix beam-search workload at its stated size -------------------------
def test_shared_prefix_16x4_full_size():
    """16 groups x 4 beams, a 1024-token prompt shared by every beam of its
    group (64 blocks at refcount 4) and tails of 1-256 tokens, stepped the way
    the benchmark steps it: beam reselection, one appended slot per beam with
    copy-on-write where siblings share a partial block, pa_copy_blocks, then
    the grouped fused write + decode over the whole batch.  The C++ block
    manager and the oracle's model run in lockstep (slots, copy pairs and
    tables identical), caches stay bit-identical to the oracle's, and every
    (beam, head) row matches the float64 oracle within the f16 tolerance --
    the grouped call and the plain fused call alike.  Each group's shared
    prefix is staged per step as the benchmark does: the prompt plus the tail
    blocks its beams inherited from a common ancestor.  The segment call
    (every block read once, whichever beams share it) matches too.

    Source: "大模型推理引擎优化：KV Cache 与连续批处理" 4.2 and
    "LLM推理引擎深度实战：从PagedAttention到分布式推理部署" 2.2 (shared blocks
    by refcount, copied on write)."""
    from oracle.allocator import BlockAllocator as OAlloc
    from oracle.cache_ops import copy_blocks as o_copy

    w = W.config_shared_prefix()
    B, beams = w.B, w.beams
    ca = ops.BlockAllocator(w.num_blocks, w.free_order)
    oa = OAlloc(w.num_blocks, w.free_order)
    roots = [10 ** 9 + g for g in range(w.groups)]
    for r in roots:
        ca.alloc_seq(r, w.prompt_len)
        oa.alloc_seq(r, w.prompt_len)
    ids = list(range(B))
    parents = [roots[i // beams] for i in range(B)]
    ca.fork_seqs(parents, ids)
    oa.fork_seqs(parents, ids)
    tails = w.tail_lens.reshape(-1)
    for i in ids:
        got = ca.append_tokens(i, int(tails[i]))
        want = oa.append_tokens(i, int(tails[i]))
        assert got == (want[0], want[1]) and want[1][0] < 0  # the prompt fills its last block
    kc, vc = w.k_pool.to(DEV), w.v_pool.to(DEV)
    okc, ovc = np_exact(w.k_pool), np_exact(w.v_pool)
    cap = -(-(w.prompt_len + int(tails.max()) + 8) // 16)
    gs_host = np.arange(0, B + 1, beams, dtype=np.int32)
    gs = torch.from_numpy(gs_host).to(DEV)
    rng = W.rng_for(23)
    q = w.q.to(DEV)
    total_cow = total_extra = total_pairs = 0
    for step in range(6):
        par = (np.arange(w.groups)[:, None] * beams + w.parents[step]).reshape(-1).tolist()
        ca.reselect(ids, par)
        oa.reselect(ids, par)
        slots, pairs = ca.append_slots(ids)
        want = oa.append_slots(ids)
        assert slots == [x[0] for x in want]
        assert pairs == [(x[1], x[2]) for x in want if x[1] >= 0]
        tables, lens = ca.tables(ids, cap)
        for i, s in enumerate(ids):
            tab, n = oa.table(s)
            assert list(tables[i][:len(tab)]) == tab and lens[i] == n
        total_cow += len(pairs)
        if pairs:
            ops.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int64, device=DEV))
            okc, ovc, _, _ = o_copy(okc, ovc, pairs)
        nk = W.randn(rng, (B, w.Hkv, w.D), torch.float16)
        nv = W.randn(rng, (B, w.Hkv, w.D), torch.float16)
        sl = torch.tensor(slots, dtype=torch.int64, device=DEV)
        bt, cl = torch.from_numpy(tables).to(DEV), torch.from_numpy(lens).to(DEV)
        ml = int(lens.max())
        # each group's shared prefix as the benchmark stages it: the prompt and
        # the tail blocks its beams inherited from a common ancestor
        pre_host = ops.shared_table_prefix(tables, lens, gs_host)
        assert (pre_host >= w.prompt_len // 16).all()
        total_extra += int((pre_host - w.prompt_len // 16).sum())
        pre = torch.from_numpy(pre_host).to(DEV)
        out = ops.decode_append_grouped(nk.to(DEV), nv.to(DEV), sl, q, kc, vc, bt, cl, ml, w.scale, gs, pre, beams,
                                        cap, out_dtype=torch.float32)
        # the plain fused call and the segment call on the same state: they
        # store the same rows again
        plain = ops.decode_append(nk.to(DEV), nv.to(DEV), sl, q, kc, vc, bt, cl, ml, w.scale,
                                  out_dtype=torch.float32)
        items, most = ops.shared_table_segments(tables, lens, gs_host)
        nm = (items[:, 3] >> 8) & 0xff
        total_pairs += int(((nm > 1) & (nm < beams)).sum())
        seg = ops.decode_append_segments(nk.to(DEV), nv.to(DEV), sl, q, kc, vc, bt, cl, ml, w.scale, gs,
                                         torch.from_numpy(items).to(DEV), beams, most, out_dtype=torch.float32)
        torch.cuda.synchronize()
        okc, ovc, _, _ = o_write(np_exact(nk), np_exact(nv), np.array(slots), okc, ovc)
        ref = paged_decode(np_exact(w.q), okc, ovc, tables, lens, w.scale)
        assert_close(out.cpu().numpy(), ref, TOL["f16"], f"grouped step {step}")
        assert_close(plain.cpu().numpy(), ref, TOL["f16"], f"plain step {step}")
        assert_close(seg.cpu().numpy(), ref, TOL["f16"], f"segments step {step}")
    assert total_cow > 0, "reselection is meant to exercise copy-on-write"
    assert total_pairs > 0, "some blocks are meant to be shared by part of a group"
    assert total_extra > 0, "some group is meant to share tail blocks beyond the prompt"
    assert np.array_equal(np_exact(kc), okc) and np.array_equal(np_exact(vc), ovc)
