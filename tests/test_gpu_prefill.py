"""GPU parity of pa_chunked_prefill (multi-token paged attention) against the
float64 oracle.

Tolerance as for decode: max-abs 2e-3 on float32 outputs for f16 / bf16
caches; 16-bit outputs within 2e-3 plus half an ulp of the output dtype.
Small ragged cases (chunks of 0 .. 130 tokens, several row tiles, ragged
tails, forced partition sizes) are compared element by element; the two
full-size workloads on sampled (token, head) rows in the launch
configuration the benchmark uses.  Shapes with more than 64 (token, head)
rows per kv head at head_dim 128 run the tcgen05 kernel, the others the
64-row mma.sync kernel; both are covered.  A prompt run as several chunks
must give bit-identical rows to one chunk where the same kernel runs (same
partition size): each row's arithmetic does not depend on the other rows of
its tile.
"""
import numpy as np
import pytest
import torch

from oracle.attention import paged_prefill
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, half_ulp, assert_close, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


@pytest.fixture(autouse=True)
def no_device_errors():
    ops.device_errors(clear=True)
    yield
    assert ops.device_errors(clear=True) == 0, "kernel flagged a device error"


def _dev_inputs(w, q_start=None, lens=None):
    qs = w.q_start if q_start is None else q_start
    lens = w.context_lens if lens is None else lens
    return (w.q.to(DEV), torch.from_numpy(np.ascontiguousarray(qs, dtype=np.int32)).to(DEV),
            w.k_pool.to(DEV), w.v_pool.to(DEV),
            torch.from_numpy(np.ascontiguousarray(w.block_tables, dtype=np.int32)).to(DEV),
            torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(DEV))


def gpu_prefill(w, out_dtype=torch.float32, split_tokens=0, q_start=None, lens=None, max_q_len=None):
    q, qs, kc, vc, bt, cl = _dev_inputs(w, q_start, lens)
    lens_np = w.context_lens if lens is None else lens
    ml = max(int(max(lens_np)), 1)
    mq = int(w.q_lens.max()) if max_q_len is None else max_q_len
    desc = ops.cache_desc(kc)
    need = int(ops.lib().pa_chunked_prefill_workspace_size(q.shape[0], len(lens_np), q.shape[1], mq, ml,
                                                          ops.C.byref(desc), split_tokens))
    # scratch starts as 0xFF bytes (NaN floats): stale rows must never leak into results
    ws = torch.full((max(need, 16),), 255, dtype=torch.uint8, device=DEV)
    out = torch.full((q.shape[0], q.shape[1], q.shape[2]), float("nan"), dtype=out_dtype, device=DEV)
    ops.chunked_prefill(q, qs, kc, vc, bt, cl, ml, mq, w.scale, out=out, workspace=ws,
                        split_tokens=split_tokens)
    torch.cuda.synchronize()
    return out.cpu()


def oracle(w, rows=None, q_start=None, lens=None):
    return paged_prefill(np_exact(w.q), w.q_start if q_start is None else q_start, np_exact(w.k_pool),
                         np_exact(w.v_pool), w.block_tables, w.context_lens if lens is None else lens,
                         w.scale, rows=rows)


SHAPES = [  # Hq, Hkv, D, kv dtype
    (4, 4, 64, "f16"), (8, 2, 128, "f16"), (8, 1, 128, "bf16"), (64, 8, 128, "bf16"),
    (32, 32, 128, "f16"), (6, 2, 64, "bf16"), (3, 1, 128, "f16"),
]
QLENS = [[1, 17, 64, 65], [130, 0, 3, 1, 40], [5, 5, 5, 5, 5, 5], [33]]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}{s[3]}")
@pytest.mark.parametrize("qi", range(len(QLENS)))
@pytest.mark.parametrize("split", [0, 16, 48])
def test_small_ragged(shape, qi, split):
    Hq, Hkv, D, dt = shape
    w = W.random_prefill_small(100 + 7 * qi + Hq, Hq, Hkv, D, dt, QLENS[qi], max_prior=90)
    ref = oracle(w)
    out = gpu_prefill(w, split_tokens=split)
    assert_close(out.numpy(), ref, TOL[dt], f"{shape} q_lens {QLENS[qi]} split {split}")


@pytest.mark.parametrize("shape", [(8, 2, 128, "f16"), (8, 1, 128, "bf16"), (4, 4, 64, "bf16")])
def test_16bit_output(shape):
    Hq, Hkv, D, dt = shape
    w = W.random_prefill_small(7, Hq, Hkv, D, dt, [70, 1, 9], max_prior=200)
    ref = oracle(w)
    out = gpu_prefill(w, out_dtype=w.q.dtype, split_tokens=64).float().numpy()
    err = np.abs(out - ref)
    assert np.all(err <= TOL[dt] + half_ulp(ref, w.q.dtype)), float(err.max())


def test_chunks_equal_one_pass_bitwise():
    """A 300-token prompt (after 37 tokens of prior context) run as chunks of
    100, 64, 1, 135 with growing context gives the rows of one 300-token pass:
    bit for bit where the chunk runs the same kernel as the whole pass (more
    than 64 (token, head) rows per kv head: the tensor-memory kernel), within
    the tolerance where it does not (the one-token chunk's 4 rows per kv head
    run the 64-row kernel)."""
    Hq, Hkv, D = 16, 4, 128
    prior = 37
    L = prior + 300
    w = W.make_prefill("p", 99, Hq, Hkv, D, "bf16", [L], [300])
    whole = gpu_prefill(w, split_tokens=64)
    done = 0
    for c in (100, 64, 1, 135):
        sub = W.PrefillWorkload("c", Hq, Hkv, D, "bf16", np.array([prior + done + c], np.int32),
                                np.array([c], np.int32), w.num_blocks, w.free_order, w.block_tables,
                                w.q[done:done + c].contiguous(), w.k_pool, w.v_pool, w.scale)
        piece = gpu_prefill(sub, split_tokens=64)
        if c * (Hq // Hkv) > 64:
            assert torch.equal(piece, whole[done:done + c]), f"chunk of {c}"
        else:
            assert_close(piece.numpy(), whole[done:done + c].numpy(), TOL["bf16"], f"chunk of {c}")
        done += c
    assert_close(whole.numpy(), oracle(w), TOL["bf16"], "one pass")


def test_single_token_chunks_match_oracle_decode_rows():
    w = W.random_prefill_small(31, 8, 2, 128, "f16", [1] * 9, max_prior=300)
    assert_close(gpu_prefill(w).numpy(), oracle(w), TOL["f16"], "one-token chunks")


def test_more_queries_than_context_gives_zero_rows_and_flags():
    w = W.random_prefill_small(41, 4, 2, 64, "f16", [20, 6], max_prior=0)
    lens = np.array([12, 6], np.int32)  # sequence 0: 20 queries, 12 keys
    out = gpu_prefill(w, lens=lens)
    assert ops.device_errors(clear=True) & ops.DEVERR_CONTEXT_LEN
    ref = oracle(w, lens=lens)
    assert_close(out.numpy(), ref, TOL["f16"], "short context")
    assert torch.count_nonzero(out[:8]) == 0


@pytest.mark.parametrize("split", [0, 16])
def test_short_queries_through_the_decode_kernel(split):
    """Up to 32 rows per kv head over a 16-bit cache run in the decode kernel,
    one grid column per query token: causal rows, a sequence with more query
    tokens than context (zero rows, flagged), an empty sequence, and the
    split-K merge of rows with different key counts."""
    w = W.random_prefill_small(47, 8, 2, 128, "f16", [4, 3, 0, 4, 1], max_prior=70)
    lens = w.context_lens.copy()
    lens[1] = 2  # 3 queries, 2 keys: its first token sees none
    out = gpu_prefill(w, lens=lens, split_tokens=split)
    assert ops.device_errors(clear=True) & ops.DEVERR_CONTEXT_LEN
    ref = oracle(w, lens=lens)
    assert_close(out.numpy(), ref, TOL["f16"], f"short queries split {split}")
    qs = w.q_start
    assert torch.count_nonzero(out[qs[1]]) == 0


def test_two_token_verify_full_size():
    """A one-draft-token verification at the speculative-verify workload's
    shapes (64 sequences, 64 q / 8 kv heads, bf16, contexts log-uniform in
    [16, 4096]) through the decode route, every row against the oracle."""
    w = W.config_spec_verify(gamma=1)
    ml = int(w.context_lens.max())
    assert ops.chunked_prefill_plan_info(w.T, w.B, w.Hq, 2, ml, w.k_pool)[1:] == \
        ops.decode_plan_info(2 * w.B, w.Hq, ml, w.k_pool)
    out = gpu_prefill(w).numpy()
    assert_close(out, oracle(w), TOL["bf16"], "two-token verify")


def test_bad_query_range_is_flagged_and_skipped():
    w = W.random_prefill_small(43, 4, 4, 64, "f16", [5, 5], max_prior=10)
    bad = np.array([0, 7, 3], np.int32)  # sequence 1 would have -4 tokens
    out = gpu_prefill(w, q_start=bad, max_q_len=8)
    assert ops.device_errors(clear=True) & ops.DEVERR_QUERY_RANGE
    ref = oracle(w, q_start=np.array([0, 7, 7]))  # sequence 0 as given; sequence 1 skipped
    assert_close(out[:7].numpy(), ref[:7], TOL["f16"], "valid sequence")
    assert torch.isnan(out[7:]).all(), "a skipped sequence's rows were written"


def test_empty_batch_and_no_tokens():
    w = W.random_prefill_small(45, 4, 4, 64, "f16", [0, 0], max_prior=10)
    out = gpu_prefill(w, max_q_len=1)
    assert out.shape[0] == 0


@pytest.mark.parametrize("name", sorted(W.PREFILL_CONFIGS))
def test_full_size_sampled(name):
    """The benchmark's workloads at full size, its launch configuration
    (library-chosen split), checked on sampled (token, head) rows that cover
    every sequence's first and last query tokens."""
    w = W.PREFILL_CONFIGS[name]()
    out = gpu_prefill(w).numpy()
    rng = np.random.Generator(np.random.PCG64(5))
    qs = w.q_start
    rows = set()
    for b in range(w.B):
        for t in (qs[b], qs[b + 1] - 1):
            rows.add((int(t), int(rng.integers(w.Hq))))
    for t in rng.integers(0, w.T, size=64):
        rows.add((int(t), int(rng.integers(w.Hq))))
    rows = sorted(rows)
    ref = oracle(w, rows=rows)
    idx = tuple(np.array(rows).T)
    assert_close(out[idx], ref[idx], TOL[w.kv_dtype], name)


@pytest.mark.parametrize("shape", [(8, 2, 128, "f16"), (8, 8, 128, "bf16"), (4, 4, 64, "f16")])
def test_stale_nan_rows_never_reach_the_output(shape):
    """Rows past each context hold NaN: weight 0, and the output stays finite
    (both kernels: 8x2 and 8x8 at head_dim 128 run the tensor-memory kernel for
    the 40-token chunk, the 64-row kernel for the 3-token one)."""
    Hq, Hkv, D, dt = shape
    w = W.random_prefill_small(71, Hq, Hkv, D, dt, [40, 3, 17], max_prior=50)
    used = np.zeros((w.num_blocks, 16), bool)
    for b in range(w.B):
        for t in range(int(w.context_lens[b])):
            used[w.block_tables[b][t // 16], t % 16] = True
    m = torch.from_numpy(~used)
    bi, ri = m.nonzero(as_tuple=True)
    w.k_pool = w.k_pool.clone()
    w.v_pool = w.v_pool.clone()
    w.k_pool[bi, :, ri, :] = float("nan")
    w.v_pool[bi, :, ri, :] = float("nan")
    assert_close(gpu_prefill(w).numpy(), oracle(w), TOL[dt], f"{shape} with NaN in unused rows")


# ---- FP8 E4M3 and INT8 caches (the 64-row kernel) ------------------------------------
def quantised_pools(w, fmt):
    """The f16 pool quantised through pa_cache_write (one token per slot):
    device codes and per-token scales."""
    N, H, _, D = w.k_pool.shape
    kin = w.k_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    vin = w.v_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(DEV)
    slots = torch.arange(N * 16, dtype=torch.int64, device=DEV)
    kc = torch.zeros((N, H, 16, D), dtype=torch.int8 if fmt == "int8" else torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((N, 16), dtype=torch.float32, device=DEV)
    vs = torch.zeros_like(ks)
    ops.cache_write(kin, vin, slots, kc, vc, ks, vs)
    torch.cuda.synchronize()
    return kc, vc, ks, vs


def gpu_prefill_q8(w, pools, out_dtype=torch.float32, split_tokens=0):
    kc, vc, ks, vs = pools
    q = w.q.to(DEV)
    qs = torch.from_numpy(np.ascontiguousarray(w.q_start, dtype=np.int32)).to(DEV)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables, dtype=np.int32)).to(DEV)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens, dtype=np.int32)).to(DEV)
    ml = max(int(w.context_lens.max()), 1)
    out = torch.full(tuple(q.shape), float("nan"), dtype=out_dtype, device=DEV)
    ops.chunked_prefill(q, qs, kc, vc, bt, cl, ml, int(w.q_lens.max()), w.scale, out=out,
                        split_tokens=split_tokens, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out.cpu()


def oracle_q8(w, pools, rows=None):
    kc, vc, ks, vs = (t.cpu().numpy() for t in pools)
    return paged_prefill(np_exact(w.q), w.q_start, kc, vc, w.block_tables, w.context_lens, w.scale,
                         k_scale=ks, v_scale=vs, rows=rows)


Q8_SHAPES = [(8, 2, "f16"), (8, 2, "bf16"), (64, 8, "bf16"), (4, 4, "f16"), (3, 1, "f16")]


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("Hq,Hkv,qdt", Q8_SHAPES)
@pytest.mark.parametrize("split", [0, 64])
def test_quantised_caches(fmt, Hq, Hkv, qdt, split):
    """1-byte caches against the oracle on the same stored codes and scales
    (chunks of 0 .. 130 tokens, row tiles with ragged tails, forced
    partitions): within the FP8 / INT8 tolerance."""
    w = W.random_prefill_small(400 + Hq + Hkv, Hq, Hkv, 128, "f16", [130, 0, 3, 1, 40, 17], max_prior=150)
    if qdt == "bf16":
        w.q = w.q.to(torch.bfloat16)
    pools = quantised_pools(w, fmt)
    assert_close(gpu_prefill_q8(w, pools, split_tokens=split).numpy(), oracle_q8(w, pools), TOL[fmt],
                 f"{fmt} {Hq}/{Hkv} {qdt} split {split}")


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_quantised_16bit_output_and_stale_rows(fmt):
    """16-bit outputs within the tolerance plus half an ulp; codes and scales
    of the rows past each context set to NaN patterns change nothing."""
    w = W.random_prefill_small(91, 16, 4, 128, "f16", [33, 5, 64], max_prior=60)
    kc, vc, ks, vs = quantised_pools(w, fmt)
    ref = oracle_q8(w, (kc, vc, ks, vs))
    used = np.zeros((w.num_blocks, 16), bool)
    for b in range(w.B):
        for t in range(int(w.context_lens[b])):
            used[w.block_tables[b][t // 16], t % 16] = True
    bi, ri = torch.from_numpy(~used).nonzero(as_tuple=True)
    bi, ri = bi.to(DEV), ri.to(DEV)
    kc.view(torch.uint8)[bi, :, ri, :] = 0x7F  # E4M3 NaN (a finite INT8 code)
    vc.view(torch.uint8)[bi, :, ri, :] = 0x7F
    ks[bi, ri] = float("nan")
    vs[bi, ri] = float("nan")
    out = gpu_prefill_q8(w, (kc, vc, ks, vs), out_dtype=torch.float16).float().numpy()
    err = np.abs(out - ref)
    assert np.all(err <= TOL[fmt] + half_ulp(ref, torch.float16)), float(np.nanmax(err))


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("q_lens,max_prior", [([1] * 6, 9000), ([1, 0, 40, 1, 1, 7], 6000), ([1, 1, 0, 1], 2500)])
def test_quantised_one_token_rows(fmt, q_lens, max_prior):
    """Over a 1-byte cache the one-token sequences of a call are served by the
    decode kernel (its query / output row is q_start[b]) and the rest by the
    multi-token kernel.  Decode-only batches, mixed batches with empty
    sequences before the one-token rows, and contexts long enough for the
    in-kernel merge (<= 8 partitions) and the merge kernel (more): every row
    within the FP8 / INT8 tolerance of the oracle on the same stored codes."""
    w = W.random_prefill_small(520 + len(q_lens) + max_prior, 16, 4, 128, "f16", q_lens, max_prior=max_prior)
    pools = quantised_pools(w, fmt)
    assert_close(gpu_prefill_q8(w, pools).numpy(), oracle_q8(w, pools), TOL[fmt],
                 f"{fmt} q_lens {q_lens} prior <= {max_prior}")
