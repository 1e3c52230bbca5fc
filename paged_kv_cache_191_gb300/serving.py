"""Iteration loop of a continuous-batching server over the paged KV cache.

A thin owner of buffers around the native engine (pa_serve_*): every
iteration one C call runs the scheduler step, stages its decisions in pinned
memory, copies them to the device in one transfer and enqueues, on one
stream, the swap-out copies of preempted requests, the decode items' cache
write fused into paged decode, the prompt chunks' cache write and
multi-token attention, and the swap-in copies of returning requests.  The
model around attention is not part of this library: queries and new K/V
rows come from caller-provided device buffers (row t for the t-th new token
of the iteration, decodes first).  The cache is 16-bit (the model's dtype)
or 1-byte codes with per-token scales (kv_dtype torch.uint8: FP8 E4M3,
torch.int8: INT8), whose scales the engine moves with every write and swap.
"""
import ctypes as C

import numpy as np
import torch

from . import ops


class ServingLoop:
    def __init__(self, num_blocks, host_blocks, num_kv_heads, num_q_heads, head_dim, dtype, max_batch,
                 max_tokens, max_context, device="cuda", free_order=None, split_tokens=0, kv_dtype=None):
        L = ops.lib()
        self.sched = ops.Scheduler(num_blocks, max_batch, max_tokens, host_blocks, free_order)
        self.Hq, self.Hkv, self.D, self.dtype, self.dev = num_q_heads, num_kv_heads, head_dim, dtype, device
        self.max_batch, self.max_tokens = max_batch, max_tokens
        self.cap = -(-max_context // 16)
        self.max_context = self.cap * 16
        self.split = split_tokens or 1024
        kv_dtype = kv_dtype or dtype
        self.q8 = kv_dtype in (torch.uint8, torch.int8)
        shape = (num_blocks, num_kv_heads, 16, head_dim)
        self.k_cache = torch.zeros(shape, dtype=kv_dtype, device=device)
        self.v_cache = torch.zeros(shape, dtype=kv_dtype, device=device)
        hshape = (max(host_blocks, 1), num_kv_heads, 16, head_dim)
        self.k_host = torch.zeros(hshape, dtype=kv_dtype).pin_memory()
        self.v_host = torch.zeros(hshape, dtype=kv_dtype).pin_memory()
        scales = [None] * 4
        if self.q8:
            self.k_scale = torch.zeros((num_blocks, 16), dtype=torch.float32, device=device)
            self.v_scale = torch.zeros_like(self.k_scale)
            self.k_host_scale = torch.zeros((max(host_blocks, 1), 16), dtype=torch.float32).pin_memory()
            self.v_host_scale = torch.zeros_like(self.k_host_scale).pin_memory()
            scales = [self.k_scale.data_ptr(), self.v_scale.data_ptr(),
                      self.k_host_scale.data_ptr() if host_blocks else None,
                      self.v_host_scale.data_ptr() if host_blocks else None]
        self.desc = ops.cache_desc(self.k_cache)
        h = self.sched._h
        self.meta_bytes = int(L.pa_serve_staging_bytes(h, self.max_context))
        ws = int(L.pa_serve_workspace_bytes(h, num_q_heads, self.max_context, C.byref(self.desc), self.split))
        self.staging_host = torch.zeros(2 * self.meta_bytes, dtype=torch.uint8).pin_memory()
        self.staging_dev = torch.zeros(self.meta_bytes, dtype=torch.uint8, device=device)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        b = ops.ServeBuffers(self.k_cache.data_ptr(), self.v_cache.data_ptr(),
                             self.k_host.data_ptr() if host_blocks else None,
                             self.v_host.data_ptr() if host_blocks else None,
                             host_blocks, num_q_heads, self.max_context, self.split,
                             self.staging_host.data_ptr(), self.staging_dev.data_ptr(), self.ws.data_ptr(), ws,
                             *scales)
        e = C.c_void_p()
        ops._check(L.pa_serve_create(h, C.byref(self.desc), C.byref(b), C.byref(e)), "pa_serve_create")
        self._e, self._L = e, L
        self.out = torch.empty((max_batch + max_tokens, num_q_heads, head_dim), dtype=dtype, device=device)
        self._dt = ops._TORCH_DT[dtype]

    def __del__(self):
        e = getattr(self, "_e", None)
        if e is not None and e.value:
            self._L.pa_serve_destroy(e)
            self._e = None

    def add(self, rid, prompt_len, max_new_tokens):
        self.sched.add(rid, prompt_len, max_new_tokens)

    def idle(self):
        return self.sched.idle()

    def plan(self):
        """Schedule the next iteration (host only); returns its token count T.
        The decisions stay in the scheduler's arrays until the next plan."""
        T = C.c_int64()
        ops._check(self._L.pa_serve_plan(self._e, C.byref(self.sched._o), C.byref(T)), "pa_serve_plan")
        return T.value

    def launch(self, q, k_new, v_new, stream=None):
        """Enqueue the planned iteration's device work (rows 0..T-1 of q,
        k_new, v_new; output rows 0..T-1 of self.out)."""
        stream = stream or torch.cuda.current_stream()
        ops._check(self._L.pa_serve_launch(self._e, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), self._dt,
                                           self.out.data_ptr(), stream.cuda_stream), "pa_serve_launch")

    def step(self, q, k_new, v_new, stream=None, attn_events=None, decisions=True):
        """plan() + launch(); returns decisions() (or, with decisions=False,
        only the token counts).  attn_events, if given, bracket the
        iteration's device work."""
        stream = stream or torch.cuda.current_stream()
        T = self.plan()
        if attn_events is not None:
            attn_events[0].record(stream)
        self.launch(q, k_new, v_new, stream)
        if attn_events is not None:
            attn_events[1].record(stream)
        if not decisions:
            return {"T": T, "n_items": self.sched._o.n_items}
        return self.decisions()

    def decisions(self):
        """The planned iteration's decisions as host arrays, with the block
        tables and context lengths of its requests and the output view
        [T, Hq, D] (valid once the stream has run the iteration)."""
        s, o = self.sched, self.sched._o
        n, T = o.n_items, int(o.n_slots)
        ids = list(s._ids[:n])
        tables, ctx = s.tables(ids, self.cap) if n else (np.zeros((0, self.cap), np.int32), np.zeros(0, np.int32))
        return {"ids": ids, "kinds": np.array(s._kinds[:n], dtype=np.int32),
                "starts": np.array(s._starts[:n], dtype=np.int32), "lens": np.array(s._lens[:n], dtype=np.int32),
                "T": T, "slots": np.array(s._slots[:T], dtype=np.int64),
                "swap_out": np.array(s._out[:2 * o.n_swap_out], dtype=np.int64).reshape(-1, 2),
                "swap_in": np.array(s._in[:2 * o.n_swap_in], dtype=np.int64).reshape(-1, 2),
                "finished": list(s._fin[:o.n_finished]), "recomputed": list(s._rec[:o.n_recomputed]),
                "tables": tables, "context_lens": ctx, "out": self.out[:T]}
