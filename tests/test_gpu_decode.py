"""GPU parity of pa_decode against the float64 oracle.

Tolerances: max-abs 2e-3 for f16/bf16 caches and 2e-2 for FP8 / INT8 caches, judged
on float32 outputs (a bf16 output alone carries up to 2^-9 relative rounding,
which exceeds 2e-3 near |o| = 1); the 16-bit outputs are checked within the
tolerance plus half an ulp of the output dtype.  Small ragged cases are
compared element by element; the full-size workloads on every
(sequence, head) row, in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

from oracle.attention import paged_decode
from oracle.cache_ops import cache_write as oracle_cache_write
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, half_ulp, assert_close, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


def gpu_decode(w, out_dtype=torch.float32, split_tokens=0, tables=None, lens=None, pools=None,
               scales=(None, None), max_len=None):
    tables = w.block_tables if tables is None else tables
    lens = w.context_lens if lens is None else lens
    kp, vp = (w.k_pool, w.v_pool) if pools is None else pools
    q = w.q.to(DEV)
    kc, vc = kp.to(DEV), vp.to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(tables, dtype=np.int32)).to(DEV)
    cl = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(DEV)
    ks = scales[0].to(DEV) if scales[0] is not None else None
    vs = scales[1].to(DEV) if scales[1] is not None else None
    ml = int(max(lens)) if max_len is None else max_len
    # scratch starts as 0xFF bytes (NaN floats): stale rows must never leak into results
    need = ops.decode_workspace_size(q.shape[0], q.shape[1], ml, kc, split_tokens)
    ws = torch.full((max(need, 16),), 255, dtype=torch.uint8, device=DEV)
    out = ops.decode(q, kc, vc, bt, cl, ml, w.scale, out_dtype=out_dtype, k_scale=ks, v_scale=vs,
                     workspace=ws, split_tokens=split_tokens)
    torch.cuda.synchronize()
    return out.cpu()


def oracle(w, heads=None, tables=None, lens=None, pools=None, scales=(None, None)):
    tables = w.block_tables if tables is None else tables
    lens = w.context_lens if lens is None else lens
    kp, vp = (w.k_pool, w.v_pool) if pools is None else pools
    return paged_decode(np_exact(w.q), np_exact(kp), np_exact(vp), tables, lens, w.scale,
                        k_scale=None if scales[0] is None else np_exact(scales[0]),
                        v_scale=None if scales[1] is None else np_exact(scales[1]), heads=heads)


def check_out_dtype(w, ref, split_tokens=0, **kw):
    """The 16-bit output: within tol + half an ulp of the output dtype."""
    out = gpu_decode(w, out_dtype=w.q.dtype, split_tokens=split_tokens, **kw).float().numpy()
    tol = TOL[w.kv_dtype]
    err = np.abs(out - ref)
    assert np.all(err <= tol + half_ulp(ref, w.q.dtype)), float(err.max())


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0, "kernel flagged a device error"


def test_tiny_workload():
    w = W.config_tiny()
    ref = oracle(w)
    assert_close(gpu_decode(w).numpy(), ref, TOL["f16"], "tiny f32 out")
    check_out_dtype(w, ref)


SHAPES = [  # Hq, Hkv, D, kv dtype
    (4, 4, 64, "f16"), (8, 2, 128, "f16"), (8, 1, 128, "bf16"), (64, 8, 128, "bf16"),
    (32, 8, 128, "f16"), (2, 2, 128, "f16"), (16, 2, 64, "bf16"), (3, 1, 128, "f16"),
]


@pytest.mark.parametrize("Hq,Hkv,D,dt", SHAPES)
@pytest.mark.parametrize("split", [0, 16, 64, 256])
def test_random_ragged(Hq, Hkv, D, dt, split):
    w = W.random_small(300 + Hq * 7 + Hkv + D, B=6, Hq=Hq, Hkv=Hkv, D=D, kv_dtype=dt, max_len=700)
    ref = oracle(w)
    assert_close(gpu_decode(w, split_tokens=split).numpy(), ref, TOL[dt], f"{Hq}/{Hkv}/{D}/{dt}/s{split}")
    if split == 0:
        check_out_dtype(w, ref)


EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000, 1024]


@pytest.mark.parametrize("dt,Hq,Hkv", [("f16", 4, 4), ("bf16", 16, 2)])
@pytest.mark.parametrize("split", [0, 256])
def test_edge_lengths(dt, Hq, Hkv, split):
    w = W.make_decode("edge", 77, len(EDGE_LENS), Hq, Hkv, 128, dt, EDGE_LENS, pool_factor=1.1)
    ref = oracle(w)
    out = gpu_decode(w, split_tokens=split).numpy()
    assert_close(out, ref, TOL[dt], "edge lengths")
    assert not out[0].any(), "empty context must give a zero row"


def test_one_token_context_returns_v_exactly():
    w = W.make_decode("one", 5, 3, 8, 2, 128, "f16", [1, 1, 1])
    out = gpu_decode(w).numpy()
    for b in range(3):
        blk = w.block_tables[b, 0]
        for h in range(8):
            assert np.array_equal(out[b, h], np_exact(w.v_pool)[blk, h // 4, 0].astype(np.float32))


def test_physical_relabelling_is_bit_identical():
    w = W.random_small(41, B=5, Hq=8, Hkv=2, D=128, kv_dtype="bf16", max_len=900)
    rng = np.random.Generator(np.random.PCG64(2))
    pi = rng.permutation(w.num_blocks)
    kp = torch.empty_like(w.k_pool)
    vp = torch.empty_like(w.v_pool)
    kp[torch.from_numpy(pi)] = w.k_pool
    vp[torch.from_numpy(pi)] = w.v_pool
    tab2 = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1)
    a = gpu_decode(w).numpy()
    b = gpu_decode(w, tables=tab2, pools=(kp, vp)).numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dt,tol", [("bf16", 1e-5), ("f16", 1e-4)])
def test_split_invariance(dt, tol):
    """Partitioning changes only the order of fp32 sums and, for f16, the
    reference maximum each p = exp(s - m) is rounded to f16 against (relative
    error <= 2^-11 per weight, about 1e-5 on outputs at these lengths); bf16 P
    is carried as hi + lo (<= 2^-17)."""
    w = W.random_small(42, B=4, Hq=16, Hkv=2, D=128, kv_dtype=dt, max_len=3000, min_len=1500)
    a = gpu_decode(w, split_tokens=16).numpy()
    b = gpu_decode(w, split_tokens=1024).numpy()
    c = gpu_decode(w).numpy()
    assert np.abs(a - b).max() <= tol and np.abs(a - c).max() <= tol


def test_constant_values_give_constant_output():
    w = W.random_small(43, B=4, Hq=8, Hkv=8, D=64, kv_dtype="f16", max_len=600)
    ones = torch.full_like(w.v_pool, 1.5)
    out = gpu_decode(w, pools=(w.k_pool, ones)).numpy()
    live = w.context_lens > 0
    assert np.abs(out[live] - 1.5).max() <= 1e-6


def test_bad_block_id_is_flagged_not_faulted():
    w = W.random_small(44, B=2, Hq=4, Hkv=4, D=64, kv_dtype="f16", max_len=60, min_len=40)
    tab = w.block_tables.copy()
    tab[1, 1] = w.num_blocks + 5
    gpu_decode(w, tables=tab)
    assert ops.device_errors(clear=True) & ops.DEVERR_BLOCK_RANGE
    lens = w.context_lens.copy()
    lens[0] = 10 ** 6
    gpu_decode(w, lens=lens, max_len=int(w.context_lens.max()))
    assert ops.device_errors(clear=True) & ops.DEVERR_CONTEXT_LEN


# ---- FP8 E4M3 caches ---------------------------------------------------------------
def fp8_pool_gpu(w):
    """Quantise the whole f16 pool through pa_cache_write (one token per slot)."""
    N, H, _, D = w.k_pool.shape
    kin = w.k_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    vin = w.v_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    slots = torch.arange(N * 16, dtype=torch.int64, device=DEV)
    kc = torch.zeros((N, H, 16, D), dtype=torch.int8 if w.kv_dtype == "int8" else torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((N, 16), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    ops.cache_write(kin, vin, slots, kc, vc, ks, vs)
    torch.cuda.synchronize()
    return kc.cpu(), vc.cpu(), ks.cpu(), vs.cpu()


def fp8_pool_oracle(w, blocks=None):
    """The oracle's own quantisation of the listed blocks (all by default)."""
    N, H, _, D = w.k_pool.shape
    blocks = np.arange(N) if blocks is None else np.asarray(sorted(set(blocks)))
    slots = (blocks[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
    kin = np_exact(w.k_pool[torch.from_numpy(blocks)]).transpose(0, 2, 1, 3).reshape(-1, H, D)
    vin = np_exact(w.v_pool[torch.from_numpy(blocks)]).transpose(0, 2, 1, 3).reshape(-1, H, D)
    kc = np.zeros((N, H, 16, D), np.int8 if w.kv_dtype == "int8" else np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((N, 16), np.float32)
    vs = np.zeros_like(ks)
    return oracle_cache_write(kin, vin, slots, kc, vc, ks, vs), blocks


@pytest.mark.parametrize("qdt", ["f16", "bf16"])
@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_fp8_small(qdt, split, fmt):
    w = W.random_small(51, B=5, Hq=16, Hkv=4, D=128, kv_dtype=fmt, max_len=800)
    if qdt == "bf16":
        w.q = w.q.to(torch.bfloat16)
    kc, vc, ks, vs = fp8_pool_gpu(w)
    (okc, ovc, oks, ovs), _ = fp8_pool_oracle(w)
    assert np.array_equal(kc.numpy(), okc) and np.array_equal(vc.numpy(), ovc)
    assert np.array_equal(ks.numpy(), oks) and np.array_equal(vs.numpy(), ovs)
    ref = paged_decode(np_exact(w.q), okc, ovc, w.block_tables, w.context_lens, w.scale, oks, ovs)
    got = gpu_decode(w, split_tokens=split, pools=(kc, vc), scales=(ks, vs)).numpy()
    assert_close(got, ref, TOL[fmt], f"{fmt} q={qdt}")
    # against the unquantised cache: reported, loosely bounded at small contexts
    ref16 = oracle(w)
    assert np.abs(got - ref16).max() < 0.25


@pytest.mark.parametrize("qscale", [300.0, 1e-3, 0.0])
@pytest.mark.parametrize("qdt", ["f16", "bf16"])
def test_fp8_query_range(qscale, qdt):
    """Over an E4M3 cache, query rows far outside E4M3's range (|q| up to
    ~1200, beyond its 448) or deep in its subnormals (|q| ~ 1e-3), and
    all-zero rows, match the oracle: Q stays in its own 16-bit type and only
    the cache's codes are converted."""
    w = W.random_small(53, B=4, Hq=16, Hkv=4, D=128, kv_dtype="fp8", max_len=300)
    q = w.q.float() * qscale
    q[1, 3] = 0.0  # one all-zero row among the others
    w.q = q.to(torch.bfloat16 if qdt == "bf16" else torch.float16)
    kc, vc, ks, vs = fp8_pool_gpu(w)
    (okc, ovc, oks, ovs), _ = fp8_pool_oracle(w)
    ref = paged_decode(np_exact(w.q), okc, ovc, w.block_tables, w.context_lens, w.scale, oks, ovs)
    got = gpu_decode(w, pools=(kc, vc), scales=(ks, vs)).numpy()
    assert np.isfinite(got).all()
    assert_close(got, ref, TOL["fp8"], f"q x {qscale} {qdt}")


# ---- full-size workloads, every row ------------------------------------------------
@pytest.mark.parametrize("cfg", ["llama7b_b32", "gqa70b_b64", "longctx_b8_f16"])
def test_full_size_all_rows(cfg):
    """Every (sequence, head) row of the full workload, in the launch
    configuration the benchmark uses (automatic partitioning)."""
    w = W.CONFIGS[cfg]()
    got = gpu_decode(w).numpy()
    assert_close(got, oracle(w), TOL[w.kv_dtype], w.name)


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_full_size_fp8_longctx_all_rows(fmt):
    """The long-context workload over a 1-byte cache: the whole pool
    quantised by pa_cache_write; each sequence's blocks quantised again by
    the oracle (in a compact pool, spawn workers) must give the same codes
    and scales bit for bit, and every row must match the oracle on those
    codes within the FP8 / INT8 tolerance, and the unquantised oracle
    within the same bound."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import os
    from tests.oracle_quant import quantise_blocks

    w = W.config_longctx(fmt)
    kc, vc, ks, vs = fp8_pool_gpu(w)
    got = gpu_decode(w, pools=(kc, vc), scales=(ks, vs)).numpy()
    seq_blocks = [w.block_tables[b][: -(-int(w.context_lens[b]) // 16)].astype(np.int64) for b in range(w.B)]
    kp, vp = np_exact(w.k_pool), np_exact(w.v_pool)
    dtype = np.int8 if fmt == "int8" else np.uint8
    tasks = [(kp[blk], vp[blk], dtype) for blk in seq_blocks]
    workers = max(1, min(8, len(os.sched_getaffinity(0))))
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        quantised = list(ex.map(quantise_blocks, tasks))
    kcn, vcn, ksn, vsn = kc.numpy(), vc.numpy(), ks.numpy(), vs.numpy()
    for b, (blk, (okc, ovc, oks, ovs)) in enumerate(zip(seq_blocks, quantised)):
        assert np.array_equal(kcn[blk], okc) and np.array_equal(vcn[blk], ovc), f"codes of sequence {b}"
        assert np.array_equal(ksn[blk], oks) and np.array_equal(vsn[blk], ovs), f"scales of sequence {b}"
        table = np.arange(len(blk), dtype=np.int64)[None, :]
        lens = w.context_lens[b:b + 1]
        q = np_exact(w.q[b:b + 1])
        ref = paged_decode(q, okc, ovc, table, lens, w.scale, oks, ovs)[0]
        assert_close(got[b], ref, TOL[fmt], f"{w.name} sequence {b}")
        ref16 = paged_decode(q, kp[blk], vp[blk], table, lens, w.scale)[0]
        assert_close(got[b], ref16, TOL[fmt], f"{w.name} sequence {b} vs unquantised")


@pytest.mark.parametrize("kv", ["f16", "bf16", "fp8", "int8"])
def test_stale_nan_rows_never_reach_the_output(kv):
    """Cache rows past each context (the tail of its last block, and blocks
    no table names) hold NaN bit patterns, as an uninitialised pool may: they
    carry weight 0 and must not turn the output into NaN."""
    D = 128
    w = W.random_small(61, B=6, Hq=8, Hkv=2, D=D, kv_dtype=kv, max_len=200, min_len=1)
    used = np.zeros((w.num_blocks, 16), bool)
    for b in range(w.B):
        n = int(w.context_lens[b])
        for t in range(n):
            used[w.block_tables[b][t // 16], t % 16] = True
    if kv in ("fp8", "int8"):
        kc, vc, ks, vs = fp8_pool_gpu(w)
        (okc, ovc, oks, ovs), _ = fp8_pool_oracle(w)
        nan_code = 0x7F  # E4M3 NaN; for INT8 any code is finite, the scale carries the NaN
        kc, vc, ks, vs = kc.clone(), vc.clone(), ks.clone(), vs.clone()
        m = torch.from_numpy(~used)
        kc.view(torch.uint8)[m.nonzero(as_tuple=True)[0], :, m.nonzero(as_tuple=True)[1], :] = nan_code
        vc.view(torch.uint8)[m.nonzero(as_tuple=True)[0], :, m.nonzero(as_tuple=True)[1], :] = nan_code
        ks[m] = float("nan")
        vs[m] = float("nan")
        got = gpu_decode(w, pools=(kc, vc), scales=(ks, vs)).numpy()
        ref = paged_decode(np_exact(w.q), okc, ovc, w.block_tables, w.context_lens, w.scale, oks, ovs)
    else:
        kp, vp = w.k_pool.clone(), w.v_pool.clone()
        m = torch.from_numpy(~used)
        bi, ri = m.nonzero(as_tuple=True)
        kp[bi, :, ri, :] = float("nan")
        vp[bi, :, ri, :] = float("nan")
        got = gpu_decode(w, pools=(kp, vp)).numpy()
        ref = oracle(w, pools=(kp, vp))
    assert_close(got, ref, TOL[kv], f"{kv} with NaN in unused rows")


@pytest.mark.parametrize("B,max_len,split", [(300, 300, 64), (5, 1100, 16), (70, 900, 64)])
def test_item_mappings(B, max_len, split):
    """Split launches over many sequences (300), many partitions (69 of 16
    tokens) and a mix (70 sequences, 15 partitions), every seventh sequence
    empty: the (sequence x kv head, partition) grid against the oracle."""
    w = W.random_small(900 + B, B=B, Hq=4, Hkv=2, D=64, kv_dtype="f16", max_len=max_len)
    lens = w.context_lens.copy()
    lens[::7] = 0
    ref = oracle(w, lens=lens)
    assert_close(gpu_decode(w, split_tokens=split, lens=lens, max_len=max_len).numpy(), ref, TOL["f16"],
                 f"B={B} split={split}")
