"""Cache write and block copy, plain NumPy (test infrastructure only).

Cache write: the decode step stores the new token's K/V in the slot its
sequence was given ([LLM-INF] 2.2, on-demand allocation: pages exist only for
generated tokens; [KV-CB] 三, append_slot).  slot s addresses block s // 16,
row s % 16 of the [num_blocks, Hkv, 16, D] cache.  A negative slot is a
padding row and is skipped (a reading: the pages are silent on padding).

FP8 variant ([LLM-INF] 5.3 allows per-channel or per-token scales; the
reading taken is one float32 scale per token per tensor, over all Hkv*D
values of that token):

    amax  = max |x|                         (float32, exact)
    scale = fl32(amax / 448)  or 1.0 when amax == 0
    code  = E4M3_RNE_satfinite( fl32(x / scale) )

where fl32 is an IEEE float32 round-to-nearest division.

INT8 variant ([LLM-INF] 5.3 names INT8 beside FP8 for the KV cache, at
per-channel or per-token granularity; the reading taken is the FP8 one --
one float32 scale per token per tensor -- with symmetric integer codes):

    scale = fl32(amax / 127)  or 1.0 when amax == 0
    code  = clamp( round_half_even( fl32(x / scale) ), -127, 127 )   (int8)

and the stored value is code * scale.  The cache dtype tells the formats
apart: uint8 caches hold E4M3 codes, int8 caches hold INT8 codes.

Block copy ([LLM-INF] 2.2 copy-on-write; [KV-CB] 4.2): for each (src, dst)
pair the whole K block, V block and, for FP8, the 16 scales of each are
copied.  Pairs must not write a block that another pair reads or writes.
"""
import numpy as np

from .fp8_e4m3 import e4m3_encode, E4M3_MAX

BLOCK_SIZE = 16


def fp8_quantize_rows(x):
    """Quantise each row of x [T, ...] -> (uint8 codes [T, ...], float32 scales [T]).

    Row t is one token (all its heads and dims): amax over the row, scale =
    fl32(amax / 448) (1.0 for an all-zero row), codes = E4M3(fl32(x / scale)).
    """
    xf = np.asarray(x, dtype=np.float32)
    T = xf.shape[0]
    flat = xf.reshape(T, -1)
    amax = np.abs(flat).max(axis=1) if flat.shape[1] else np.zeros(T, np.float32)
    scale = np.where(amax == 0, np.float32(1.0),
                     amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    y = (flat / scale[:, None]).astype(np.float32)
    return e4m3_encode(y).reshape(xf.shape), scale


INT8_MAX = 127


def int8_quantize_rows(x):
    """Quantise each row of x [T, ...] -> (int8 codes [T, ...], float32 scales [T]).

    Row t is one token: amax over the row, scale = fl32(amax / 127) (1.0 for
    an all-zero row), codes = round-half-even(fl32(x / scale)) clamped to
    [-127, 127] (the clamp only guards the rounding of the scale).
    """
    xf = np.asarray(x, dtype=np.float32)
    T = xf.shape[0]
    flat = xf.reshape(T, -1)
    amax = np.abs(flat).max(axis=1) if flat.shape[1] else np.zeros(T, np.float32)
    scale = np.where(amax == 0, np.float32(1.0),
                     amax.astype(np.float32) / np.float32(INT8_MAX)).astype(np.float32)
    y = (flat / scale[:, None]).astype(np.float32)
    codes = np.clip(np.rint(y), -INT8_MAX, INT8_MAX).astype(np.int8)  # rint: ties to even
    return codes.reshape(xf.shape), scale


def quantize_rows(x, cache_dtype):
    """Per-token quantiser of a cache's format: uint8 -> E4M3, int8 -> INT8."""
    return int8_quantize_rows(x) if np.dtype(cache_dtype) == np.int8 else fp8_quantize_rows(x)


def fp8_quantize_token(x):
    """Quantise one token's values (any shape) -> (uint8 codes, float32 scale)."""
    codes, scale = fp8_quantize_rows(np.asarray(x)[None])
    return codes[0], np.float32(scale[0])


def cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None):
    """Return new (k_cache, v_cache, k_scale, v_scale) after writing T tokens.

    k, v: [T, Hkv, D] (float16/float32 values); caches: [num_blocks, Hkv, 16, D]
    in the storage dtype (float16, float32 holding bf16 values, or uint8 E4M3 /
    int8 codes when k_scale/v_scale [num_blocks, 16] float32 are given).
    """
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    fp8 = k_scale is not None
    if fp8:
        k_scale = np.array(k_scale, dtype=np.float32, copy=True)
        v_scale = np.array(v_scale, dtype=np.float32, copy=True)
    slots = np.asarray(slot_mapping).astype(np.int64)
    used = slots[slots >= 0]
    if len(np.unique(used)) != len(used):
        raise ValueError("duplicate slots in one cache write")
    nslots = k_cache.shape[0] * BLOCK_SIZE
    if (slots >= nslots).any():
        raise ValueError("slot out of range")
    idx = np.nonzero(slots >= 0)[0]
    for c0 in range(0, len(idx), 4096):          # chunks bound the float64 temporaries
        rows = idx[c0:c0 + 4096]
        blk, off = slots[rows] // BLOCK_SIZE, slots[rows] % BLOCK_SIZE
        if fp8:
            kc, ks = quantize_rows(np.asarray(k)[rows], k_cache.dtype)
            vc, vs = quantize_rows(np.asarray(v)[rows], v_cache.dtype)
            k_cache[blk, :, off, :] = kc
            v_cache[blk, :, off, :] = vc
            k_scale[blk, off] = ks
            v_scale[blk, off] = vs
        else:
            k_cache[blk, :, off, :] = np.asarray(k)[rows]
            v_cache[blk, :, off, :] = np.asarray(v)[rows]
    return k_cache, v_cache, k_scale, v_scale


def copy_blocks(k_cache, v_cache, pairs, k_scale=None, v_scale=None):
    """Return new caches with block dst := block src for each (src, dst) pair."""
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    srcs, dsts = pairs[:, 0], pairs[:, 1]
    if len(np.unique(dsts)) != len(dsts) or np.intersect1d(srcs, dsts).size:
        raise ValueError("copy pairs overlap: a dst repeats or is also a src")
    k_new = np.array(k_cache, copy=True)
    v_new = np.array(v_cache, copy=True)
    ks = None if k_scale is None else np.array(k_scale, copy=True)
    vs = None if v_scale is None else np.array(v_scale, copy=True)
    for s, d in pairs:
        k_new[d] = k_cache[s]
        v_new[d] = v_cache[s]
        if ks is not None:
            ks[d] = k_scale[s]
            vs[d] = v_scale[s]
    return k_new, v_new, ks, vs


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, dst_ks=None, dst_vs=None, src_ks=None, src_vs=None):
    """Return new dst pools with dst block d := src block s for each (s, d).

    Preemption moves a request's pages between the GPU cache and a CPU pool
    ([LLM-INF] 3.2); both pools are laid out like a cache.  No dst may repeat.
    """
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    if len(np.unique(pairs[:, 1])) != len(pairs):
        raise ValueError("a dst block repeats")
    k_new, v_new = np.array(dst_k, copy=True), np.array(dst_v, copy=True)
    ks = None if dst_ks is None else np.array(dst_ks, copy=True)
    vs = None if dst_vs is None else np.array(dst_vs, copy=True)
    for s, d in pairs:
        k_new[d] = src_k[s]
        v_new[d] = src_v[s]
        if ks is not None:
            ks[d] = src_ks[s]
            vs[d] = src_vs[s]
    return k_new, v_new, ks, vs
