"""Python binding of libpagedkv.so (argument marshalling only).

Every device step runs in the library's CUDA kernels; this module checks
tensor device/dtype/shape/contiguity, passes raw pointers and the current
torch stream through the C ABI declared in include/pagedkv.h, and turns a
non-zero pa_status into an exception.  PyTorch is used for device memory and
streams only.  There is no fallback: if the library is missing, every call
raises.
"""
import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_NOT_FOUND, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = range(6)
F16, BF16, FP8_E4M3, F32, INT8 = 0, 1, 2, 3, 4
BLOCK_SIZE = 16
DEVERR_SLOT_RANGE, DEVERR_BLOCK_RANGE, DEVERR_CONTEXT_LEN, DEVERR_TIMEOUT = 1, 2, 4, 8
DEVERR_QUERY_RANGE = 16
DEVERR_GROUP = 32

_TORCH_DT = {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
             torch.uint8: FP8_E4M3, torch.float8_e4m3fn: FP8_E4M3, torch.int8: INT8}


class PagedKVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"[pa_status {status}] {msg}")
        self.status = status


class OutOfBlocks(PagedKVError):
    pass


class UnknownSequence(PagedKVError):
    pass


class CacheDesc(C.Structure):
    _fields_ = [("num_blocks", C.c_int32), ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("block_size", C.c_int32), ("kv_dtype", C.c_int32)]


_P = C.c_void_p
_I32, _I64, _U64, _F = C.c_int32, C.c_int64, C.c_uint64, C.c_float
_I32P, _I64P, _U64P = C.POINTER(C.c_int32), C.POINTER(C.c_int64), C.POINTER(C.c_uint64)

# name -> (restype, argtypes); mirrors include/pagedkv.h
class SchedStepOut(C.Structure):
    _fields_ = [("n_items", C.c_int32), ("ids", C.POINTER(C.c_uint64)), ("kinds", C.POINTER(C.c_int32)),
                ("starts", C.POINTER(C.c_int32)), ("lens", C.POINTER(C.c_int32)),
                ("n_slots", C.c_int64), ("slots", C.POINTER(C.c_int64)),
                ("n_finished", C.c_int32), ("finished", C.POINTER(C.c_uint64)),
                ("n_swap_out", C.c_int32), ("swap_out", C.POINTER(C.c_int64)),
                ("n_swap_in", C.c_int32), ("swap_in", C.POINTER(C.c_int64)),
                ("n_recomputed", C.c_int32), ("recomputed", C.POINTER(C.c_uint64))]


class ServeBuffers(C.Structure):
    _fields_ = [("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("k_host", C.c_void_p), ("v_host", C.c_void_p),
                ("host_blocks", C.c_int32), ("num_q_heads", C.c_int32), ("max_context", C.c_int32),
                ("split_tokens", C.c_int32), ("staging_host", C.c_void_p), ("staging_dev", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
                ("k_scale", C.c_void_p), ("v_scale", C.c_void_p), ("k_host_scale", C.c_void_p),
                ("v_host_scale", C.c_void_p)]


SIGNATURES = {
    "pa_last_error": (C.c_char_p, []),
    "pa_version": (_I32, []),
    "pa_cache_write": (C.c_int, [_P, _P, _I32, _P, _I64, _P, _P, _P, _P, C.POINTER(CacheDesc), _P]),
    "pa_decode_workspace_size": (C.c_size_t, [_I32, _I32, _I32, C.POINTER(CacheDesc), _I32]),
    "pa_decode_plan_info": (C.c_int, [_I32, _I32, _I32, C.POINTER(CacheDesc), _I32, _I32P, _I32P, _I32P]),
    "pa_chunked_prefill_plan_info": (C.c_int, [_I32, _I32, _I32, _I32, _I32, C.POINTER(CacheDesc), _I32,
                                               _I32P, _I32P, _I32P, _I32P]),
    "pa_decode": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _F, _P, _I32,
                            C.POINTER(CacheDesc), _P, C.c_size_t, _I32, _P]),
    "pa_decode_append": (C.c_int, [_P, _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                   _I32, _F, _P, _I32, C.POINTER(CacheDesc), _P, C.c_size_t, _I32, _P]),
    "pa_decode_static_ws": (C.c_int, [_P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _F, _P,
                                      _I32, C.POINTER(CacheDesc), _I32, _P]),
    "pa_decode_grouped_workspace_size": (C.c_size_t, [_I32, _I32, _I32, _I32, _I32, _I32, C.POINTER(CacheDesc),
                                                      _I32]),
    "pa_decode_append_grouped": (C.c_int, [_P, _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                           _I32, _F, _P, _P, _I32, _I32, _I32, _P, _I32, C.POINTER(CacheDesc),
                                           _P, C.c_size_t, _I32, _P]),
    "pa_decode_segments_workspace_size": (C.c_size_t, [_I32, _I32, _I32, _I32, _I32, C.POINTER(CacheDesc)]),
    "pa_decode_append_segments": (C.c_int, [_P, _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32,
                                            _I32, _I32, _F, _P, _I32, _I32, _P, _I32, _I32, _P, _I32,
                                            C.POINTER(CacheDesc), _P, C.c_size_t, _P]),
    "pa_table_segments": (C.c_int, [_P, _I32, _P, _P, _I32, _I32, _P, _I32, _P, _P]),
    "pa_decode_items_plan": (C.c_int, [_P, _I32, _I32, _I32, C.POINTER(CacheDesc), _I32, _I32P, _I32P, _I32P]),
    "pa_chunked_prefill_workspace_size": (C.c_size_t, [_I32, _I32, _I32, _I32, _I32, C.POINTER(CacheDesc),
                                                       _I32]),
    "pa_chunked_prefill": (C.c_int, [_P, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                     _F, _P, _I32, C.POINTER(CacheDesc), _P, C.c_size_t, _I32, _P]),
    "pa_copy_blocks": (C.c_int, [_P, _P, _P, _P, _P, _I64, C.POINTER(CacheDesc), _P]),
    "pa_swap_blocks": (C.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _I32, _P, _I64,
                                 C.POINTER(CacheDesc), _P]),
    "pa_device_errors": (C.c_int, [C.POINTER(C.c_uint32), _I32]),
    "pa_alloc_create": (C.c_int, [_I32, _I32, _I64P, C.POINTER(_P)]),
    "pa_alloc_destroy": (None, [_P]),
    "pa_alloc_seq": (C.c_int, [_P, _U64, _I64]),
    "pa_append_slot": (C.c_int, [_P, _U64, _I64P, _I64P, _I64P]),
    "pa_append_slots": (C.c_int, [_P, _U64P, _I32, _I64P, _I64P, _I32P]),
    "pa_append_tokens": (C.c_int, [_P, _U64, _I64, _I64P, _I64P, _I64P]),
    "pa_fork": (C.c_int, [_P, _U64, _U64]),
    "pa_fork_seqs": (C.c_int, [_P, _U64P, _U64P, _I32]),
    "pa_free_seqs": (C.c_int, [_P, _U64P, _I32]),
    "pa_reselect": (C.c_int, [_P, _U64P, _I32P, _I32]),
    "pa_free_seq": (C.c_int, [_P, _U64]),
    "pa_block_table": (C.c_int, [_P, _U64, _I32P, _I32, _I32P, _I64P]),
    "pa_block_tables": (C.c_int, [_P, _U64P, _I32, _I32P, _I32, _I32P]),
    "pa_alloc_stats": (C.c_int, [_P, _I32P, _I32P, _I32P]),
    "pa_sched_create": (C.c_int, [_I32, _I64P, _I32, _I32, _I32, C.POINTER(_P)]),
    "pa_sched_destroy": (None, [_P]),
    "pa_sched_add": (C.c_int, [_P, _U64, _I32, _I32]),
    "pa_sched_step": (C.c_int, [_P, C.POINTER(SchedStepOut)]),
    "pa_sched_allocator": (_P, [_P]),
    "pa_sched_stats": (C.c_int, [_P, _I32P, _I32P, _I32P, _I32P, _I32P]),
    "pa_sched_limits": (C.c_int, [_P, _I32P, _I32P, _I32P]),
    "pa_serve_staging_bytes": (C.c_size_t, [_P, _I32]),
    "pa_serve_workspace_bytes": (C.c_size_t, [_P, _I32, _I32, C.POINTER(CacheDesc), _I32]),
    "pa_serve_create": (C.c_int, [_P, C.POINTER(CacheDesc), C.POINTER(ServeBuffers), C.POINTER(_P)]),
    "pa_serve_destroy": (None, [_P]),
    "pa_serve_plan": (C.c_int, [_P, C.POINTER(SchedStepOut), _I64P]),
    "pa_serve_launch": (C.c_int, [_P, _P, _P, _P, _I32, _P, _P]),
    "pa_serve_step": (C.c_int, [_P, _P, _P, _P, _I32, _P, C.POINTER(SchedStepOut), _P]),
    "pa_free_list": (C.c_int, [_P, _I32P, _I32, _I32P]),
}

_lib = None


def lib():
    """Load libpagedkv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_191_gb300.build` (needs nvcc)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status, what=""):
    if status == PA_OK:
        return
    msg = lib().pa_last_error().decode(errors="replace")
    cls = {PA_ERR_OOM: OutOfBlocks, PA_ERR_NOT_FOUND: UnknownSequence}.get(status, PagedKVError)
    raise cls(status, f"{what}: {msg}" if what else msg)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dev(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def kv_dtype_of(cache):
    if cache.dtype not in _TORCH_DT or cache.dtype == torch.float32:
        raise ValueError(f"unsupported cache dtype {cache.dtype}")
    return _TORCH_DT[cache.dtype]


def cache_desc(k_cache):
    """CacheDesc of a [num_blocks, Hkv, 16, D] cache tensor."""
    if k_cache.dim() != 4 or k_cache.shape[2] != BLOCK_SIZE:
        raise ValueError("cache must be [num_blocks, num_kv_heads, 16, head_dim]")
    nb, h, _, d = k_cache.shape
    return CacheDesc(nb, h, d, BLOCK_SIZE, kv_dtype_of(k_cache))


def cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None, stream=None):
    """Store rows k, v [T, Hkv, D] at slot_mapping [T] (int64; <0 skips)."""
    for t, n in ((k, "k"), (v, "v"), (slot_mapping, "slot_mapping"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache differ")
    T = k.shape[0]
    if k.shape != (T, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise ValueError("k, v must be [T, num_kv_heads, head_dim]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [T]")
    if k.dtype != v.dtype or k.dtype not in (torch.float16, torch.bfloat16, torch.float32):
        raise ValueError("k, v must share dtype f16 / bf16 / f32")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if t is not None:
            _dev(t, n)
    _check(lib().pa_cache_write(_ptr(k), _ptr(v), _TORCH_DT[k.dtype], _ptr(slot_mapping), T,
                                _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                C.byref(desc), _stream(stream)), "pa_cache_write")


def decode_plan_info(B, num_q_heads, max_context_len, k_cache, split_tokens=0):
    """(partitions, blocks per partition, kernels launched) of a decode call."""
    desc = cache_desc(k_cache)
    p, bpp, k = C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().pa_decode_plan_info(B, num_q_heads, max_context_len, C.byref(desc), split_tokens, C.byref(p),
                                     C.byref(bpp), C.byref(k)), "pa_decode_plan_info")
    return p.value, bpp.value, k.value


def chunked_prefill_plan_info(num_tokens, B, num_q_heads, max_q_len, max_context_len, k_cache, split_tokens=0):
    """(tensor cores, partitions, blocks per partition, kernels launched) of a multi-token call."""
    desc = cache_desc(k_cache)
    tc, p, bpp, k = C.c_int32(), C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().pa_chunked_prefill_plan_info(num_tokens, B, num_q_heads, max_q_len, max_context_len, C.byref(desc),
                                              split_tokens, C.byref(tc), C.byref(p), C.byref(bpp), C.byref(k)),
           "pa_chunked_prefill_plan_info")
    return tc.value, p.value, bpp.value, k.value


def decode_workspace_size(B, num_q_heads, max_context_len, k_cache, split_tokens=0):
    desc = cache_desc(k_cache)
    return int(lib().pa_decode_workspace_size(B, num_q_heads, max_context_len, C.byref(desc), split_tokens))


def decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
           out=None, out_dtype=None, k_scale=None, v_scale=None, workspace=None,
           split_tokens=0, stream=None):
    """Paged decode attention; returns out [B, Hq, D] (q dtype, or out_dtype)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    if D != desc.head_dim:
        raise ValueError("q head_dim differs from the cache")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be int32 [B, max_blocks]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != B:
        raise ValueError("context_lens must be int32 [B]")
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=odt, device=q.device)
    else:
        _dev(out, "out")
        if out.shape != (B, Hq, D):
            raise ValueError("out must be [B, Hq, D]")
        odt = out.dtype
    need = int(lib().pa_decode_workspace_size(B, Hq, max_context_len, C.byref(desc), split_tokens))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode(_ptr(q), _TORCH_DT[q.dtype], _ptr(k_cache), _ptr(v_cache),
                           _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
                           _ptr(context_lens), int(max_context_len), B, Hq, float(scale),
                           _ptr(out), _TORCH_DT[odt], C.byref(desc), _ptr(workspace), ws_bytes,
                           int(split_tokens), _stream(stream)), "pa_decode")
    return out


def chunked_prefill(q, q_start, k_cache, v_cache, block_tables, context_lens, max_context_len,
                    max_q_len, scale, out=None, out_dtype=None, workspace=None, split_tokens=0,
                    stream=None, k_scale=None, v_scale=None):
    """Multi-token paged attention (chunked prefill / speculative verify).

    q: [T, Hq, D] packed query tokens; q_start: int32 [B + 1] offsets;
    k_scale, v_scale: float32 [num_blocks, 16] for FP8 / INT8 caches.
    Returns out [T, Hq, D] (q dtype, or out_dtype).
    """
    for t, n in ((q, "q"), (q_start, "q_start"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    T, Hq, D = q.shape
    B = context_lens.numel()
    if D != desc.head_dim:
        raise ValueError("q head_dim differs from the cache")
    if q_start.dtype != torch.int32 or q_start.numel() != B + 1:
        raise ValueError("q_start must be int32 [B + 1]")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be int32 [B, max_blocks]")
    if context_lens.dtype != torch.int32:
        raise ValueError("context_lens must be int32 [B]")
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((T, Hq, D), dtype=odt, device=q.device)
    else:
        _dev(out, "out")
        if out.shape != (T, Hq, D):
            raise ValueError("out must be [T, Hq, D]")
        odt = out.dtype
    need = int(lib().pa_chunked_prefill_workspace_size(T, B, Hq, int(max_q_len), int(max_context_len),
                                                       C.byref(desc), int(split_tokens)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_chunked_prefill(_ptr(q), _TORCH_DT[q.dtype], _ptr(q_start), T, int(max_q_len),
                                    _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(block_tables), block_tables.shape[1],
                                    _ptr(context_lens), int(max_context_len), B, Hq, float(scale),
                                    _ptr(out), _TORCH_DT[odt], C.byref(desc), _ptr(workspace), ws_bytes,
                                    int(split_tokens), _stream(stream)), "pa_chunked_prefill")
    return out


def decode_append(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables, context_lens,
                  max_context_len, scale, out=None, out_dtype=None, k_scale=None, v_scale=None,
                  workspace=None, split_tokens=0, stream=None):
    """cache_write(k_new, v_new, slot_mapping) fused into decode (one launch)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (slot_mapping, "slot_mapping"), (q, "q"),
                 (k_cache, "k_cache"), (v_cache, "v_cache"), (block_tables, "block_tables"),
                 (context_lens, "context_lens")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    if k_new.shape != (B, desc.num_kv_heads, D) or v_new.shape != k_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new, v_new must be [B, num_kv_heads, head_dim] of one dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be int64 [B]")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be int32 [B, max_blocks]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != B:
        raise ValueError("context_lens must be int32 [B]")
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=odt, device=q.device)
    else:
        _dev(out, "out")
        odt = out.dtype
    need = int(lib().pa_decode_workspace_size(B, Hq, max_context_len, C.byref(desc), split_tokens))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode_append(_ptr(k_new), _ptr(v_new), _TORCH_DT[k_new.dtype], _ptr(slot_mapping),
                                  _ptr(q), _TORCH_DT[q.dtype], _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                  _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                  int(max_context_len), B, Hq, float(scale), _ptr(out), _TORCH_DT[odt],
                                  C.byref(desc), _ptr(workspace), ws_bytes, int(split_tokens), _stream(stream)),
           "pa_decode_append")
    return out


def decode_append_grouped(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables, context_lens,
                          max_context_len, scale, group_start, prefix_blocks, max_group_size, max_prefix_blocks,
                          out=None, out_dtype=None, k_scale=None, v_scale=None, workspace=None, split_tokens=0,
                          stream=None):
    """decode_append with shared-prefix groups: group k is sequences
    group_start[k] .. group_start[k+1]-1 (int32 [n_groups + 1], device),
    sharing their first prefix_blocks[k] blocks (int32 [n_groups], device);
    each shared tile is read once for the whole group."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (slot_mapping, "slot_mapping"), (q, "q"),
                 (k_cache, "k_cache"), (v_cache, "v_cache"), (block_tables, "block_tables"),
                 (context_lens, "context_lens"), (group_start, "group_start"), (prefix_blocks, "prefix_blocks")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    n_groups = group_start.numel() - 1
    if group_start.dtype != torch.int32 or prefix_blocks.dtype != torch.int32 or prefix_blocks.numel() != n_groups:
        raise ValueError("group_start must be int32 [n_groups + 1], prefix_blocks int32 [n_groups]")
    if k_new.shape != (B, desc.num_kv_heads, D) or v_new.shape != k_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new, v_new must be [B, num_kv_heads, head_dim] of one dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be int64 [B]")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be int32 [B, max_blocks]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != B:
        raise ValueError("context_lens must be int32 [B]")
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=odt, device=q.device)
    else:
        _dev(out, "out")
        odt = out.dtype
    need = int(lib().pa_decode_grouped_workspace_size(B, Hq, int(max_context_len), n_groups, int(max_group_size),
                                                      int(max_prefix_blocks), C.byref(desc), int(split_tokens)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode_append_grouped(
        _ptr(k_new), _ptr(v_new), _TORCH_DT[k_new.dtype], _ptr(slot_mapping), _ptr(q), _TORCH_DT[q.dtype],
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), B, Hq, float(scale), _ptr(group_start), _ptr(prefix_blocks),
        n_groups, int(max_group_size), int(max_prefix_blocks), _ptr(out), _TORCH_DT[odt], C.byref(desc),
        _ptr(workspace), ws_bytes, int(split_tokens), _stream(stream)), "pa_decode_append_grouped")
    return out


def decode_append_segments(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale, group_start, items, max_group_size, max_group_items,
                           out=None, out_dtype=None, k_scale=None, v_scale=None, workspace=None, stream=None):
    """decode_append over groups whose members share blocks in any pattern:
    items (int32 [n_items, 4], device) lists the runs of table positions a
    subset of a group's members all hold, each with its partial slot
    (shared_table_segments builds them).  Each block is read once for every
    member that holds it."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (slot_mapping, "slot_mapping"), (q, "q"),
                 (k_cache, "k_cache"), (v_cache, "v_cache"), (block_tables, "block_tables"),
                 (context_lens, "context_lens"), (group_start, "group_start"), (items, "items")):
        _dev(t, n)
    desc = cache_desc(k_cache)
    B, Hq, D = q.shape
    n_groups = group_start.numel() - 1
    if group_start.dtype != torch.int32:
        raise ValueError("group_start must be int32 [n_groups + 1]")
    if items.dtype != torch.int32 or items.dim() != 2 or items.shape[1] != 4:
        raise ValueError("items must be int32 [n_items, 4]")
    if k_new.shape != (B, desc.num_kv_heads, D) or v_new.shape != k_new.shape or k_new.dtype != v_new.dtype:
        raise ValueError("k_new, v_new must be [B, num_kv_heads, head_dim] of one dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be int64 [B]")
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be int32 [B, max_blocks]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != B:
        raise ValueError("context_lens must be int32 [B]")
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=odt, device=q.device)
    else:
        _dev(out, "out")
        odt = out.dtype
    need = int(lib().pa_decode_segments_workspace_size(B, Hq, n_groups, int(max_group_size), int(max_group_items),
                                                       C.byref(desc)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode_append_segments(
        _ptr(k_new), _ptr(v_new), _TORCH_DT[k_new.dtype], _ptr(slot_mapping), _ptr(q), _TORCH_DT[q.dtype],
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), B, Hq, float(scale), _ptr(group_start), n_groups,
        int(max_group_size), _ptr(items), items.shape[0], int(max_group_items), _ptr(out),
        _TORCH_DT[odt], C.byref(desc), _ptr(workspace), ws_bytes, _stream(stream)), "pa_decode_append_segments")
    return out


def shared_table_segments(block_tables, context_lens, group_start, blocks_per_item=40):
    """Host helper for decode_append_segments (pa_table_segments): the items
    of the groups.  At table position j, the members of a group whose blocks
    there are the same physical block form a class (a member alone at and
    after its last block, which takes this step's token); a segment is a
    maximal run of positions over which a class stays the same, cut into
    items of at most blocks_per_item (<= 64) blocks.  A group's items take
    slots 0, 1, ... in the order (lowest member, position); the list is
    sorted longest first.  block_tables int [B, max_blocks], context_lens int
    [B], group_start int [n + 1].  Returns (items int32 [n_items, 4] =
    {group, member list (4 bits per member index), first block,
    n_blocks | n_members << 8 | slot << 16}, the most slots of one group)."""
    import numpy as np
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    gs = np.ascontiguousarray(group_start, dtype=np.int32)
    if tables.ndim != 2 or lens.shape != (tables.shape[0],):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    n = len(gs) - 1
    if n < 0 or (n > 0 and (gs[0] < 0 or gs[-1] > tables.shape[0])):
        raise ValueError("group_start out of range")
    cap = int(((lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE).sum()) + 1
    items = np.empty((cap, 4), dtype=np.int32)
    count, most = C.c_int32(), C.c_int32()
    st = lib().pa_table_segments(tables.ctypes.data_as(C.c_void_p), tables.shape[1], lens.ctypes.data_as(C.c_void_p),
                                 gs.ctypes.data_as(C.c_void_p), n, int(blocks_per_item),
                                 items.ctypes.data_as(C.c_void_p), cap, C.byref(count), C.byref(most))
    if st != PA_OK:
        raise ValueError(lib().pa_last_error().decode())
    return items[:count.value].copy(), most.value


def decode_items_plan(context_lens, num_q_heads, max_context_len, k_cache, split_tokens=0):
    """pa_decode_items_plan: (use_items, blocks_per_item, max_items_per_seq)
    for a batch without shared blocks, from its host context lengths.
    use_items says whether decode_append_segments over one-member groups
    (the sequences' live partitions, shared_table_segments with group_start
    0..B) beats decode_append's fixed grid: fewer than half of that grid's
    cells hold blocks."""
    import numpy as np
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    desc = cache_desc(k_cache)
    use, bpi, most = C.c_int32(), C.c_int32(), C.c_int32()
    _check(lib().pa_decode_items_plan(lens.ctypes.data_as(C.c_void_p), lens.shape[0], num_q_heads, max_context_len,
                                      C.byref(desc), split_tokens, C.byref(use), C.byref(bpi), C.byref(most)),
           "pa_decode_items_plan")
    return bool(use.value), bpi.value, most.value


def prefix_groups(block_tables, context_lens, max_group_size):
    """Host helper for decode_append_grouped: split the batch, in order, into
    groups of consecutive sequences that share leading table entries (the
    beams of one prompt after fork), at most max_group_size long.

    block_tables int [B, max_blocks], context_lens int [B] (host arrays).  A
    group's prefix counts the leading entries every member holds equally
    among the whole blocks before each member's last token (the part the
    grouped decode may share).  A sequence joins the group before it while
    that keeps the shared prefix at least one block; every other sequence
    starts a group.  Returns (group_start int32 [n + 1], prefix_blocks int32
    [n])."""
    import numpy as np
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens, dtype=np.int64)
    B = len(lens)
    if max_group_size < 1:
        raise ValueError("max_group_size must be >= 1")
    usable = np.where(lens > 0, (lens - 1) // BLOCK_SIZE, 0)  # whole blocks before the last token
    starts, prefixes = [], []
    b = 0
    while b < B:
        g0, pre = b, int(usable[b])
        b += 1
        while b < B and b - g0 < max_group_size:
            lim = min(pre, int(usable[b]))
            same = tables[g0, :lim] == tables[b, :lim]
            common = int(lim if same.all() else np.argmin(same))
            if common < 1:
                break
            pre = common
            b += 1
        starts.append(g0)
        prefixes.append(pre if b - g0 > 1 else 0)
    starts.append(B)
    return np.asarray(starts, dtype=np.int32), np.asarray(prefixes, dtype=np.int32)


def shared_table_prefix(block_tables, context_lens, group_start, out=None):
    """Host helper for decode_append_grouped over fixed groups (the beams of
    one prompt): for each group, the number of leading table entries that all
    of its members hold, counted up to the longest member's blocks.  The
    kernel clamps it further to the whole blocks before each member's last
    token.  block_tables int [B, max_blocks], context_lens int [B],
    group_start int [n + 1]; returns (or fills `out`) int32 [n]."""
    import numpy as np
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens)
    gs = np.asarray(group_start)
    n = len(gs) - 1
    res = np.zeros(n, dtype=np.int32) if out is None else out
    sizes = np.diff(gs)
    if n and (sizes == sizes[0]).all() and sizes[0] > 0:  # equal groups: one vectorised pass
        k = int(sizes[0])
        nblk = int((int(lens[gs[0]:gs[-1]].max()) + BLOCK_SIZE - 1) // BLOCK_SIZE) if gs[-1] > gs[0] else 0
        t = tables[gs[0]:gs[-1], :nblk].reshape(n, k, nblk)
        same = (t == t[:, :1, :]).all(axis=1)
        res[:] = np.where(same.all(axis=1), nblk, np.argmin(same, axis=1))
        return res
    for i in range(n):
        a, b = int(gs[i]), int(gs[i + 1])
        if b <= a:
            res[i] = 0
            continue
        nblk = int((int(lens[a:b].max()) + BLOCK_SIZE - 1) // BLOCK_SIZE)
        same = (tables[a:b, :nblk] == tables[a, :nblk]).all(axis=0)
        res[i] = nblk if same.all() else int(np.argmin(same))
    return res


def copy_blocks(k_cache, v_cache, pairs, k_scale=None, v_scale=None, stream=None):
    """Copy whole blocks for each (src, dst) row of pairs (int64 [n, 2])."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (pairs, "pairs")):
        _dev(t, n)
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [n, 2]")
    desc = cache_desc(k_cache)
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _ptr(pairs), pairs.shape[0], C.byref(desc), _stream(stream)),
           "pa_copy_blocks")


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, dst_k_scale=None, dst_v_scale=None,
                src_k_scale=None, src_v_scale=None, stream=None):
    """Copy blocks pairs[i] = (src, dst) from pool (src_k, src_v) to (dst_k, dst_v).

    Pools are [num_blocks, Hkv, 16, D] tensors on the GPU or in pinned host
    memory; pairs is an int64 [n, 2] tensor on the GPU or pinned."""
    for t, n in ((dst_k, "dst_k"), (dst_v, "dst_v"), (src_k, "src_k"), (src_v, "src_v"), (pairs, "pairs")):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous tensor")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be on the GPU or in pinned host memory")
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [n, 2]")
    if dst_k.shape[1:] != src_k.shape[1:] or dst_k.dtype != src_k.dtype:
        raise ValueError("pools differ in shape or dtype")
    desc = cache_desc(src_k)
    _check(lib().pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(dst_k_scale), _ptr(dst_v_scale), dst_k.shape[0],
                                _ptr(src_k), _ptr(src_v), _ptr(src_k_scale), _ptr(src_v_scale), src_k.shape[0],
                                _ptr(pairs), pairs.shape[0], C.byref(desc), _stream(stream)), "pa_swap_blocks")


def device_errors(clear=True):
    """Device error word (DEVERR_* bits); synchronises the device."""
    flags = C.c_uint32(0)
    _check(lib().pa_device_errors(C.byref(flags), 1 if clear else 0), "pa_device_errors")
    return flags.value


class BlockAllocator:
    """Host block manager (C++): FIFO free list, block tables, refcounts, CoW."""

    def __init__(self, num_blocks, free_order=None):
        h = C.c_void_p()
        order = None
        if free_order is not None:
            self._order = (C.c_int64 * num_blocks)(*[int(x) for x in free_order])
            order = C.cast(self._order, _I64P)
        _check(lib().pa_alloc_create(num_blocks, BLOCK_SIZE, order, C.byref(h)), "pa_alloc_create")
        self._h = h
        self.num_blocks = num_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pa_alloc_destroy(h)
            self._h = None

    def alloc_seq(self, seq_id, num_tokens):
        _check(lib().pa_alloc_seq(self._h, seq_id, num_tokens), "pa_alloc_seq")

    def append_slot(self, seq_id):
        s, a, b = C.c_int64(), C.c_int64(), C.c_int64()
        _check(lib().pa_append_slot(self._h, seq_id, C.byref(s), C.byref(a), C.byref(b)), "pa_append_slot")
        return s.value, a.value, b.value

    def append_slots(self, seq_ids):
        """-> (slots list, [(src, dst), ...])"""
        n = len(seq_ids)
        ids = (C.c_uint64 * max(n, 1))(*seq_ids)
        slots = (C.c_int64 * max(n, 1))()
        pairs = (C.c_int64 * max(2 * n, 2))()
        nc = C.c_int32()
        _check(lib().pa_append_slots(self._h, ids, n, slots, pairs, C.byref(nc)), "pa_append_slots")
        return list(slots[:n]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(nc.value)]

    def append_slots_into(self, ids, n, slots, pairs, n_cow):
        """Zero-copy variant over caller-owned ctypes/numpy buffers (pointers)."""
        _check(lib().pa_append_slots(self._h, ids, n, slots, pairs, n_cow), "pa_append_slots")

    def append_tokens(self, seq_id, n, want_slots=True):
        """-> (slots list or None, (cow_src, cow_dst))"""
        buf = (C.c_int64 * max(n, 1))() if want_slots else None
        a, b = C.c_int64(), C.c_int64()
        _check(lib().pa_append_tokens(self._h, seq_id, n, buf, C.byref(a), C.byref(b)), "pa_append_tokens")
        return (list(buf[:n]) if want_slots else None), (a.value, b.value)

    def fork(self, parent, child):
        _check(lib().pa_fork(self._h, parent, child), "pa_fork")

    def fork_seqs(self, parents, children):
        n = len(parents)
        P = (C.c_uint64 * max(n, 1))(*parents)
        Q = (C.c_uint64 * max(n, 1))(*children)
        _check(lib().pa_fork_seqs(self._h, P, Q, n), "pa_fork_seqs")

    def reselect(self, ids, parent_idx):
        n = len(ids)
        A = (C.c_uint64 * max(n, 1))(*[int(x) for x in ids])
        P = (C.c_int32 * max(n, 1))(*[int(x) for x in parent_idx])
        _check(lib().pa_reselect(self._h, A, P, n), "pa_reselect")

    def free_seqs(self, ids):
        n = len(ids)
        A = (C.c_uint64 * max(n, 1))(*ids)
        _check(lib().pa_free_seqs(self._h, A, n), "pa_free_seqs")

    def free_seq(self, seq_id):
        _check(lib().pa_free_seq(self._h, seq_id), "pa_free_seq")

    def table(self, seq_id):
        nb, nt = C.c_int32(), C.c_int64()
        _check(lib().pa_block_table(self._h, seq_id, None, 0, C.byref(nb), C.byref(nt)), "pa_block_table")
        buf = (C.c_int32 * max(nb.value, 1))()
        _check(lib().pa_block_table(self._h, seq_id, buf, nb.value, C.byref(nb), C.byref(nt)), "pa_block_table")
        return list(buf[:nb.value]), nt.value

    def tables(self, seq_ids, cap):
        """-> (tables int32 [n][cap] as nested lists, context_lens list)"""
        import numpy as np
        n = len(seq_ids)
        ids = (C.c_uint64 * max(n, 1))(*seq_ids)
        tab = np.empty((max(n, 1), cap), dtype=np.int32)
        lens = np.empty(max(n, 1), dtype=np.int32)
        _check(lib().pa_block_tables(self._h, ids, n, tab.ctypes.data_as(_I32P), cap,
                                     lens.ctypes.data_as(_I32P)), "pa_block_tables")
        return tab[:n], lens[:n]

    def stats(self):
        tot, fr = C.c_int32(), C.c_int32()
        rc = (C.c_int32 * self.num_blocks)()
        _check(lib().pa_alloc_stats(self._h, C.byref(tot), C.byref(fr), rc), "pa_alloc_stats")
        return tot.value, fr.value, list(rc)

    def free_list(self):
        n = C.c_int32()
        _check(lib().pa_free_list(self._h, None, 0, C.byref(n)), "pa_free_list")
        buf = (C.c_int32 * max(n.value, 1))()
        _check(lib().pa_free_list(self._h, buf, n.value, C.byref(n)), "pa_free_list")
        return list(buf[:n.value])

    def utilization(self):
        tot, fr, _ = self.stats()
        return (tot - fr) / tot


class Scheduler:
    """Continuous-batching scheduler (C++) over its own block manager.

    step() -> (items, finished, swap_out, swap_in, recomputed) with items as
    (id, "prefill" | "decode", start position, [slots]) in batch order and
    the pairs as (from block, to block) tuples.
    """

    def __init__(self, num_blocks, max_batch, max_tokens, host_blocks, free_order=None):
        h = C.c_void_p()
        order = None
        if free_order is not None:
            self._order = (C.c_int64 * num_blocks)(*[int(x) for x in free_order])
            order = C.cast(self._order, _I64P)
        _check(lib().pa_sched_create(num_blocks, order, max_batch, max_tokens, host_blocks, C.byref(h)),
               "pa_sched_create")
        self._h = h
        self.num_blocks, self.max_batch, self.max_tokens = num_blocks, max_batch, max_tokens
        nb, nt = max_batch, max_batch + max_tokens
        self._ids, self._kinds = (C.c_uint64 * nb)(), (C.c_int32 * nb)()
        self._starts, self._lens = (C.c_int32 * nb)(), (C.c_int32 * nb)()
        self._slots = (C.c_int64 * nt)()
        self._fin, self._rec = (C.c_uint64 * nb)(), (C.c_uint64 * nb)()
        self._out, self._in = (C.c_int64 * (2 * num_blocks))(), (C.c_int64 * (2 * num_blocks))()
        o = SchedStepOut()
        o.ids, o.kinds, o.starts, o.lens = self._ids, self._kinds, self._starts, self._lens
        o.slots, o.finished, o.recomputed = self._slots, self._fin, self._rec
        o.swap_out, o.swap_in = self._out, self._in
        self._o = o
        self.alloc_handle = C.c_void_p(lib().pa_sched_allocator(h))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pa_sched_destroy(h)
            self._h = None

    def add(self, rid, prompt_len, max_new_tokens):
        _check(lib().pa_sched_add(self._h, rid, prompt_len, max_new_tokens), "pa_sched_add")

    def step_raw(self):
        """Run one step; the decisions stay in the ctypes arrays of self._o."""
        _check(lib().pa_sched_step(self._h, C.byref(self._o)), "pa_sched_step")
        return self._o

    def step(self):
        o = self.step_raw()
        items, k = [], 0
        for i in range(o.n_items):
            n = o.lens[i]
            items.append((o.ids[i], "decode" if o.kinds[i] == 1 else "prefill", o.starts[i],
                          list(self._slots[k:k + n])))
            k += n
        pairs = lambda a, n: [(a[2 * i], a[2 * i + 1]) for i in range(n)]
        return (items, list(self._fin[:o.n_finished]), pairs(self._out, o.n_swap_out),
                pairs(self._in, o.n_swap_in), list(self._rec[:o.n_recomputed]))

    def stats(self):
        v = [C.c_int32() for _ in range(5)]
        _check(lib().pa_sched_stats(self._h, *[C.byref(x) for x in v]), "pa_sched_stats")
        return tuple(x.value for x in v)  # waiting, running, swapped, free blocks, free host blocks

    def idle(self):
        w, r, s, _, _ = self.stats()
        return w == 0 and r == 0 and s == 0

    def tables(self, ids, cap):
        """(int32 [n, cap] tables, int32 [n] context lengths) of running ids."""
        import numpy as np
        n = len(ids)
        tab = np.full((max(n, 1), cap), -1, dtype=np.int32)
        lens = np.zeros(max(n, 1), dtype=np.int32)
        arr = (C.c_uint64 * max(n, 1))(*ids)
        _check(lib().pa_block_tables(self.alloc_handle, arr, n, tab.ctypes.data_as(_I32P), cap,
                                     lens.ctypes.data_as(_I32P)), "pa_block_tables")
        return tab[:n], lens[:n]
