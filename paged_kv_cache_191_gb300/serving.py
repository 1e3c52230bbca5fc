"""Iteration loop of a continuous-batching server over the paged KV cache.

Each iteration the C++ scheduler decides which requests run and which new
tokens they bring; this loop turns that into device work on one stream, in
the order the decisions require:

  1. swap-out copies (GPU blocks -> pinned host pool) of preempted requests,
     before anything can overwrite the blocks they release;
  2. the cache write of every new token's K/V into its slot;
  3. multi-token paged attention over all running requests at once (prompt
     chunks and decode steps in one launch, causal inside each chunk);
  4. swap-in copies (pinned host pool -> GPU) of requests that return next
     iteration.

Every per-iteration input (slots, query offsets, context lengths, block
tables, swap pairs) goes to the device in one host-to-device copy from a
pinned staging buffer.  The model around attention is not part of this
library: queries and new K/V rows come from caller-provided device buffers.
"""
import ctypes as C

import numpy as np
import torch

from . import ops


class ServingLoop:
    def __init__(self, num_blocks, host_blocks, num_kv_heads, num_q_heads, head_dim, dtype, max_batch,
                 max_tokens, max_context, device="cuda", free_order=None, split_tokens=0):
        self.sched = ops.Scheduler(num_blocks, max_batch, max_tokens, host_blocks, free_order)
        self.Hq, self.Hkv, self.D, self.dtype, self.dev = num_q_heads, num_kv_heads, head_dim, dtype, device
        self.max_batch, self.max_tokens = max_batch, max_tokens
        self.cap = -(-max_context // 16)
        self.max_context = self.cap * 16
        shape = (num_blocks, num_kv_heads, 16, head_dim)
        self.k_cache = torch.zeros(shape, dtype=dtype, device=device)
        self.v_cache = torch.zeros(shape, dtype=dtype, device=device)
        hshape = (max(host_blocks, 1), num_kv_heads, 16, head_dim)
        self.k_host = torch.zeros(hshape, dtype=dtype).pin_memory()
        self.v_host = torch.zeros(hshape, dtype=dtype).pin_memory()
        self.split = split_tokens
        T = max_batch + max_tokens
        # staging layout (bytes): slots i64[T] | swap_out i64[2N] | swap_in i64[2N] |
        # q_start i32[B+1] | lens i32[B] | tables i32[B*cap]
        N = num_blocks
        self._off = {}
        o = 0
        for name, n, size in (("slots", T, 8), ("swap_out", 2 * N, 8), ("swap_in", 2 * N, 8),
                              ("q_start", max_batch + 1, 4), ("lens", max_batch, 4),
                              ("tables", max_batch * self.cap, 4)):
            self._off[name] = (o, n, size)
            o += -(-n * size // 16) * 16
        self.meta_bytes = o
        # two pinned staging buffers: the host fills one while the device may
        # still be copying the other (the host runs at most one step ahead)
        self.meta_hosts = [torch.zeros(o, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.meta_dev = torch.zeros(o, dtype=torch.uint8, device=device)
        self._nps = [{k: np.frombuffer((C.c_char * o).from_address(h.data_ptr()), dtype=np.uint8)
                      [a:a + n * sz].view(np.int64 if sz == 8 else np.int32) for k, (a, n, sz) in self._off.items()}
                     for h in self.meta_hosts]
        self._dv = {k: self.meta_dev[a:a + n * sz].view(torch.int64 if sz == 8 else torch.int32)
                    for k, (a, n, sz) in self._off.items()}
        desc = ops.cache_desc(self.k_cache)
        self.ws_bytes = int(ops.lib().pa_chunked_prefill_workspace_size(T, max_batch, num_q_heads, max_tokens,
                                                                        self.max_context, C.byref(desc),
                                                                        split_tokens))
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        self.out = torch.empty((T, num_q_heads, head_dim), dtype=dtype, device=device)
        self.step_no = 0

    def add(self, rid, prompt_len, max_new_tokens):
        self.sched.add(rid, prompt_len, max_new_tokens)

    def idle(self):
        return self.sched.idle()

    def step(self, q, k_new, v_new, stream=None, attn_events=None):
        """Schedule one iteration and enqueue its device work.

        q: device [>= T, Hq, D], k_new / v_new: device [>= T, Hkv, D] in the
        cache dtype, row i for the i-th new token of the iteration (items in
        batch order).  Returns a dict with the decisions (host arrays) and the
        attention output view [T, Hq, D] (valid once the stream reaches it).
        """
        stream = stream or torch.cuda.current_stream()
        o = self.sched.step_raw()
        n, T = o.n_items, int(o.n_slots)
        ids = list(o.ids[:n])
        lens = np.ctypeslib.as_array(o.lens, shape=(self.max_batch,))[:n]
        starts = np.ctypeslib.as_array(o.starts, shape=(self.max_batch,))[:n]
        m = self._nps[self.step_no & 1]
        if T:
            m["slots"][:T] = np.ctypeslib.as_array(o.slots, shape=(T,))
        if o.n_swap_out:
            m["swap_out"][:2 * o.n_swap_out] = np.ctypeslib.as_array(o.swap_out, shape=(2 * o.n_swap_out,))
        if o.n_swap_in:
            m["swap_in"][:2 * o.n_swap_in] = np.ctypeslib.as_array(o.swap_in, shape=(2 * o.n_swap_in,))
        m["q_start"][0] = 0
        np.cumsum(lens, out=m["q_start"][1:n + 1])
        tab = m["tables"][:n * self.cap]
        if n:
            arr = (C.c_uint64 * n)(*ids)
            ops._check(ops.lib().pa_block_tables(self.sched.alloc_handle, arr, n,
                                                 tab.ctypes.data_as(ops._I32P), self.cap,
                                                 m["lens"].ctypes.data_as(ops._I32P)), "pa_block_tables")
        if T:
            need = int(ops.lib().pa_chunked_prefill_workspace_size(T, n, self.Hq, int(lens.max()), self.max_context,
                                                                   C.byref(ops.cache_desc(self.k_cache)),
                                                                   self.split))
            if need > self.ws.numel():  # a smaller batch may split its contexts more finely
                self.ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
        with torch.cuda.stream(stream):
            self.meta_dev.copy_(self.meta_hosts[self.step_no & 1], non_blocking=True)
            d = self._dv
            if o.n_swap_out:
                ops.swap_blocks(self.k_host, self.v_host, self.k_cache, self.v_cache,
                                d["swap_out"][:2 * o.n_swap_out].view(-1, 2), stream=stream)
            if T:
                ops.cache_write(k_new[:T], v_new[:T], d["slots"][:T], self.k_cache, self.v_cache, stream=stream)
                if attn_events is not None:
                    attn_events[0].record(stream)
                ops.chunked_prefill(q[:T], d["q_start"][:n + 1], self.k_cache, self.v_cache,
                                    d["tables"][:n * self.cap].view(n, self.cap), d["lens"][:n],
                                    self.max_context, int(lens.max()), 1.0 / float(np.sqrt(self.D)),
                                    out=self.out[:T], workspace=self.ws, split_tokens=self.split,
                                    stream=stream)
                if attn_events is not None:
                    attn_events[1].record(stream)
            if o.n_swap_in:
                ops.swap_blocks(self.k_cache, self.v_cache, self.k_host, self.v_host,
                                d["swap_in"][:2 * o.n_swap_in].view(-1, 2), stream=stream)
        # staging buffer i % 2 is refilled two steps later: keep the host at
        # most one iteration ahead of the device
        ev = torch.cuda.Event()
        ev.record(stream)
        prev, self._pending = getattr(self, "_pending", None), ev
        if prev is not None:
            prev.synchronize()
        self.step_no += 1
        kinds = np.ctypeslib.as_array(o.kinds, shape=(self.max_batch,))[:n]
        return {"ids": ids, "kinds": kinds.copy(), "starts": starts.copy(), "lens": lens.copy(), "T": T,
                "slots": m["slots"][:T].copy(),
                "swap_out": m["swap_out"][:2 * o.n_swap_out].reshape(-1, 2).copy(),
                "swap_in": m["swap_in"][:2 * o.n_swap_in].reshape(-1, 2).copy(),
                "finished": list(o.finished[:o.n_finished]), "recomputed": list(o.recomputed[:o.n_recomputed]),
                "tables": tab.reshape(-1, self.cap)[:n].copy() if n else np.zeros((0, self.cap), np.int32),
                "out": self.out[:T]}
