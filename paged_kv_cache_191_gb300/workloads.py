"""Seeded synthetic inputs for paged decode attention.

This module only draws random inputs; it holds none of the attention,
quantisation or allocation arithmetic, and it is shared by the CUDA-path
tests, the oracle tests and the benchmark so that both sides see identical
stored values.

Every tensor is drawn N(0, 1) in float32 from a NumPy PCG64 generator and
rounded once to its storage dtype.  The five named workloads follow the
decode scenarios the paged-KV pages motivate (LLaMA-7B-shaped batch decode,
a 70B-shaped grouped-query decode, long-context split decode, shared-prefix
parallel sampling); no public dataset is involved.

Block tables are a seeded random assignment of distinct physical blocks to
each sequence's logical blocks: the pool is permuted and each sequence takes
the next ceil(L/16) ids of that permutation, so physical ids are scattered
over the pool.  The same permutation is returned as ``free_order`` so that a
block allocator whose free list starts in that order reproduces the tables.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

BLOCK = 16
SEED_BASE = 1000

KV_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


def rng_for(seed):
    return np.random.Generator(np.random.PCG64(seed))


def randn(rng, shape, dtype):
    """N(0,1) float32 draw rounded once to ``dtype`` (a torch dtype)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(dtype)


@dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str                 # "f16", "bf16", "fp8" or "int8" (fp8 / int8: pools hold the f16 source)
    context_lens: np.ndarray      # int32 [B], includes this step's new token
    num_blocks: int
    free_order: np.ndarray        # int64 permutation of the pool
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 padded
    q: torch.Tensor               # [B, Hq, D]
    k_pool: torch.Tensor          # [num_blocks, Hkv, 16, D]
    v_pool: torch.Tensor
    new_k: torch.Tensor           # [B, Hkv, D] this step's token
    new_v: torch.Tensor
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def max_blocks(self):
        return self.block_tables.shape[1]


def _tables_from_order(order, lens, max_blocks):
    tables = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-int(n) // BLOCK)
        tables[b, :nb] = order[pos:pos + nb]
        pos += nb
    return tables


def make_decode(name, seed, B, Hq, Hkv, D, kv_dtype, lens, pool_factor=1.2,
                min_pool=None, max_blocks=None):
    rng = rng_for(seed)
    lens = np.asarray(lens, dtype=np.int32)
    demand = int(sum(-(-int(n) // BLOCK) for n in lens))
    num_blocks = max(int(math.ceil(pool_factor * demand)), demand, 1)
    if min_pool is not None:
        num_blocks = max(num_blocks, min_pool)
    order = rng.permutation(num_blocks).astype(np.int64)
    mb = max_blocks or max(1, max(-(-int(n) // BLOCK) for n in lens))
    tables = _tables_from_order(order, lens, mb)
    tdt = torch.float16 if kv_dtype in ("f16", "fp8", "int8") else torch.bfloat16
    q = randn(rng, (B, Hq, D), tdt)
    k_pool = randn(rng, (num_blocks, Hkv, BLOCK, D), tdt)
    v_pool = randn(rng, (num_blocks, Hkv, BLOCK, D), tdt)
    new_k = randn(rng, (B, Hkv, D), tdt)
    new_v = randn(rng, (B, Hkv, D), tdt)
    return DecodeWorkload(name, B, Hq, Hkv, D, kv_dtype, lens, num_blocks, order, tables,
                          q, k_pool, v_pool, new_k, new_v, 1.0 / math.sqrt(D))


def config_tiny():
    """4 seqs, lens {5,17,32,47}, 4/4 heads, D=64, fp16, 32-block permuted pool."""
    return make_decode("tiny", SEED_BASE + 1, 4, 4, 4, 64, "f16", [5, 17, 32, 47],
                       pool_factor=1.0, min_pool=32)


def config_llama7b(B=32):
    """Batch 32, 32/32 heads, D=128, fp16, lens uniform in [1, 2048]."""
    rng = rng_for(SEED_BASE + 2)
    lens = rng.integers(1, 2048, size=B, endpoint=True)
    return make_decode("llama7b_b32", SEED_BASE + 2 + 100, B, 32, 32, 128, "f16", lens)


def config_gqa70b(B=64):
    """Batch 64, 64 q / 8 kv heads, D=128, bf16, lens log-uniform in [16, 4096]."""
    rng = rng_for(SEED_BASE + 3)
    lens = np.rint(np.exp(rng.uniform(math.log(16), math.log(4096), size=B))).astype(np.int64)
    return make_decode("gqa70b_b64", SEED_BASE + 3 + 100, B, 64, 8, 128, "bf16", lens)


def config_longctx(kv_dtype="f16", B=8):
    """Batch 8, 32 q / 8 kv heads, D=128, lens uniform in [16384, 32768]."""
    rng = rng_for(SEED_BASE + 4)
    lens = rng.integers(16384, 32768, size=B, endpoint=True)
    return make_decode("longctx_b8_" + kv_dtype, SEED_BASE + 4 + 100, B, 32, 8, 128, kv_dtype, lens)


@dataclass
class SharedPrefixWorkload:
    """16 groups x 4 beams sharing a 1024-token prompt, with divergent tails.

    The random choices are inputs; the block allocator turns them into
    tables, forks and copy-on-write pairs.
    """
    groups: int
    beams: int
    prompt_len: int
    tail_lens: np.ndarray         # int64 [groups, beams], each in [1, 256]
    parents: np.ndarray           # int64 [steps, groups, beams] parent beam per new beam
    Hq: int
    Hkv: int
    D: int
    num_blocks: int
    free_order: np.ndarray
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    q: torch.Tensor               # [groups*beams, Hq, D]
    new_k: torch.Tensor           # [groups*beams, Hkv, D]
    new_v: torch.Tensor
    scale: float
    name: str = "shared_prefix_16x4"
    kv_dtype: str = "f16"

    @property
    def B(self):
        return self.groups * self.beams


def config_shared_prefix(steps=64, groups=16, beams=4, prompt_len=1024, H=32, D=128):
    seed = SEED_BASE + 5
    rng = rng_for(seed)
    tails = rng.integers(1, 256, size=(groups, beams), endpoint=True)
    parents = rng.integers(0, beams, size=(steps, groups, beams))
    # demand: one prompt per group plus each beam's tail and one extra block per
    # step of headroom for copy-on-write and growth
    prompt_blocks = -(-prompt_len // BLOCK)
    tail_blocks = int(sum(-(-int(t) // BLOCK) + 1 for t in tails.ravel()))
    demand = groups * prompt_blocks + tail_blocks + groups * beams * (-(-steps // BLOCK) + 2)
    num_blocks = int(math.ceil(1.2 * demand))
    order = rng.permutation(num_blocks).astype(np.int64)
    B = groups * beams
    q = randn(rng, (B, H, D), torch.float16)
    k_pool = randn(rng, (num_blocks, H, BLOCK, D), torch.float16)
    v_pool = randn(rng, (num_blocks, H, BLOCK, D), torch.float16)
    new_k = randn(rng, (B, H, D), torch.float16)
    new_v = randn(rng, (B, H, D), torch.float16)
    return SharedPrefixWorkload(groups, beams, prompt_len, tails, parents, H, H, D,
                                num_blocks, order, k_pool, v_pool, q, new_k, new_v,
                                1.0 / math.sqrt(D))


def random_small(seed, B, Hq, Hkv, D, kv_dtype, max_len, min_len=0, extra_blocks=3):
    """Small ragged case for parity sweeps: lens uniform in [min_len, max_len]."""
    rng = rng_for(seed)
    lens = rng.integers(min_len, max_len, size=B, endpoint=True)
    return make_decode(f"rand{seed}", seed + 7, B, Hq, Hkv, D, kv_dtype, lens,
                       pool_factor=1.0, min_pool=int(sum(-(-int(n) // BLOCK) for n in lens)) + extra_blocks)


def random_slots(seed, T, num_blocks, n_skip=0):
    """T distinct random slots in the pool, with ``n_skip`` of them set to -1."""
    rng = rng_for(seed)
    slots = rng.choice(num_blocks * BLOCK, size=T, replace=False).astype(np.int64)
    if n_skip:
        slots[rng.choice(T, size=n_skip, replace=False)] = -1
    return slots


def random_pairs(seed, num_blocks, n):
    """n (src, dst) block pairs with all 2n ids distinct."""
    rng = rng_for(seed)
    ids = rng.choice(num_blocks, size=2 * n, replace=False).astype(np.int64)
    return ids.reshape(n, 2)


@dataclass
class PrefillWorkload:
    """Several query tokens per sequence: the last q_lens[b] of its context."""
    name: str
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str
    context_lens: np.ndarray      # int32 [B], includes the chunk
    q_lens: np.ndarray            # int32 [B]
    num_blocks: int
    free_order: np.ndarray
    block_tables: np.ndarray      # int32 [B, max_blocks], -1 padded
    q: torch.Tensor               # [T, Hq, D], sequences' tokens packed in order
    k_pool: torch.Tensor          # [num_blocks, Hkv, 16, D] (chunk K/V included)
    v_pool: torch.Tensor
    scale: float

    @property
    def B(self):
        return len(self.context_lens)

    @property
    def q_start(self):
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def T(self):
        return int(self.q_lens.sum())

    @property
    def G(self):
        return self.Hq // self.Hkv


def make_prefill(name, seed, Hq, Hkv, D, kv_dtype, ctx_lens, q_lens, pool_factor=1.2, extra_blocks=0):
    rng = rng_for(seed)
    lens = np.asarray(ctx_lens, dtype=np.int32)
    ql = np.asarray(q_lens, dtype=np.int32)
    demand = int(sum(-(-int(n) // BLOCK) for n in lens))
    num_blocks = max(int(math.ceil(pool_factor * demand)) + extra_blocks, 1)
    order = rng.permutation(num_blocks).astype(np.int64)
    mb = max(1, max(-(-int(n) // BLOCK) for n in lens))
    tables = _tables_from_order(order, lens, mb)
    tdt = KV_TORCH.get(kv_dtype, torch.float16)  # 1-byte caches: f16 values, quantised on the device
    q = randn(rng, (int(ql.sum()), Hq, D), tdt)
    k_pool = randn(rng, (num_blocks, Hkv, BLOCK, D), tdt)
    v_pool = randn(rng, (num_blocks, Hkv, BLOCK, D), tdt)
    return PrefillWorkload(name, Hq, Hkv, D, kv_dtype, lens, ql, num_blocks, order, tables, q,
                           k_pool, v_pool, 1.0 / math.sqrt(D))


def config_prefill_mix(chunks=4, chunk=512, decodes=28, kv="f16"):
    """LLaMA-7B shapes (32/32 heads, D=128, fp16): `chunks` prompt chunks of
    `chunk` tokens at prior contexts uniform in [0, 4096 - chunk], batched with
    `decodes` one-token decode steps at contexts uniform in [1, 2048].  kv
    "fp8" / "int8": the same values in a 1-byte cache (f16 queries)."""
    rng = rng_for(SEED_BASE + 6)
    prior = rng.integers(0, 4096 - chunk, size=chunks, endpoint=True)
    dec = rng.integers(1, 2048, size=decodes, endpoint=True)
    ctx = np.concatenate([prior + chunk, dec])
    ql = np.concatenate([np.full(chunks, chunk), np.ones(decodes, dtype=np.int64)])
    name = "prefill_mix_llama7b" + ("" if kv == "f16" else "_" + kv)
    return make_prefill(name, SEED_BASE + 6 + 100, 32, 32, 128, kv, ctx, ql)


def config_spec_verify(B=64, gamma=4):
    """GQA-70B shapes (64 q / 8 kv heads, D=128, bf16): each of B sequences
    verifies gamma draft tokens plus the bonus token (gamma + 1 queries) at
    contexts log-uniform in [16, 4096]."""
    rng = rng_for(SEED_BASE + 7)
    base = np.rint(np.exp(rng.uniform(math.log(16), math.log(4096), size=B))).astype(np.int64)
    ql = np.full(B, gamma + 1)
    return make_prefill("spec_verify_gqa70b", SEED_BASE + 7 + 100, 64, 8, 128, "bf16", base + gamma + 1, ql)


def random_prefill_small(seed, Hq, Hkv, D, kv_dtype, q_lens, max_prior=80):
    """Small ragged multi-token case: each sequence's context is its chunk
    plus a prior context uniform in [0, max_prior]."""
    rng = rng_for(seed)
    ql = np.asarray(q_lens, dtype=np.int64)
    prior = rng.integers(0, max_prior, size=len(ql), endpoint=True)
    return make_prefill(f"prefill{seed}", seed + 11, Hq, Hkv, D, kv_dtype, prior + ql, ql,
                        pool_factor=1.0, extra_blocks=3)


@dataclass
class ServingTrace:
    """Synthetic request stream for the serving loop: Poisson arrivals of
    `rate` requests per iteration, prompts log-uniform in [prompt_min,
    prompt_max], outputs uniform in [out_min, out_max]; iteration i's
    arrivals are drawn from their own seeded generator."""
    name: str
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str
    num_blocks: int
    host_blocks: int
    max_batch: int
    max_tokens: int
    rate: float
    prompt_min: int
    prompt_max: int
    out_min: int
    out_max: int
    seed: int

    @property
    def max_context(self):
        return self.prompt_max + self.out_max

    def arrivals(self, it):
        rng = rng_for(self.seed * 1_000_003 + it)
        out = []
        for j in range(int(rng.poisson(self.rate))):
            p = int(np.rint(np.exp(rng.uniform(math.log(self.prompt_min), math.log(self.prompt_max)))))
            m = int(rng.integers(self.out_min, self.out_max, endpoint=True))
            out.append((it * 1000 + j, p, m))
        return out


def serving_llama7b():
    """LLaMA-7B shapes (32/32 heads, D=128, fp16); 2048 GPU blocks (32K
    tokens, 1 GB of K+V) and 1024 host blocks for swapping; batch <= 64,
    2048 tokens per iteration; prompts 32..2048, outputs 16..512, 1.5
    arrivals per iteration (more than the pool sustains, so requests queue
    and are preempted)."""
    return ServingTrace("serving_llama7b", 32, 32, 128, "f16", 2048, 1024, 64, 2048, 1.5,
                        32, 2048, 16, 512, SEED_BASE + 8)


PREFILL_CONFIGS = {
    "prefill_mix_llama7b": config_prefill_mix,
    "prefill_mix_llama7b_fp8": lambda: config_prefill_mix(kv="fp8"),
    "spec_verify_gqa70b": config_spec_verify,
}


CONFIGS = {
    "tiny": config_tiny,
    "llama7b_b32": config_llama7b,
    "gqa70b_b64": config_gqa70b,
    "longctx_b8_f16": lambda: config_longctx("f16"),
    "longctx_b8_fp8": lambda: config_longctx("fp8"),
    "longctx_b8_int8": lambda: config_longctx("int8"),
}
