"""Decode steps with host inputs at low host overhead.

A DecodeSession binds a cache and a batch shape once.  Each step's inputs
live in one pinned host staging buffer:

    slots int64 [B] | context_lens int32 [B] | block_tables int32 [B, max_blocks]
    | q [B, Hq, D] | k_new [B, Hkv, D] | v_new [B, Hkv, D]
    | items int32 [B * max_items_per_seq, 4]   (items mode only)

(each part 16-byte aligned).  The caller fills the buffer: the block manager
writes slots, lengths and tables straight into it through the pointers that
`meta_ptrs()` returns, and the model writes q / k_new / v_new through
`inputs()`.  launch() then issues one host-to-device copy of the buffer, one
pa_decode_append launch (cache write fused into attention) and one
device-to-host copy of the output; wait() returns the output once it is on
the host (step() does both).  The ctypes arguments of the launch are built
once.  Host buffers rotate over a small ring, so the next step's buffer can
be filled (block manager, model) while the device runs the current one.

Items mode: with skewed context lengths most cells of pa_decode_append's
fixed (sequence, kv head, partition) grid hold no blocks.  Then launch()
lists the step's live partitions on the host (pa_table_segments over B
one-member groups, from the lengths and tables already in the buffer),
copies them with the rest and runs pa_decode_append_segments instead.
items="auto" decides per step (pa_decode_items_plan), True always lists,
False never does.
"""
import ctypes as C

import torch

from . import ops


def _align16(n):
    return (n + 15) & ~15


class DecodeSession:
    def __init__(self, k_cache, v_cache, batch, num_q_heads, max_blocks, max_context_len, scale,
                 dtype, k_scale=None, v_scale=None, out_dtype=None, split_tokens=0, ring=2, items="auto"):
        for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
            ops._dev(t, n)
        L = ops.lib()
        self.desc = ops.cache_desc(k_cache)
        self.B, self.Hq, self.Hkv, self.D = batch, num_q_heads, self.desc.num_kv_heads, self.desc.head_dim
        self.max_blocks, self.max_context_len = max_blocks, max_context_len
        dev = k_cache.device
        e = torch.empty((), dtype=dtype).element_size()
        B, Hq, Hkv, D = self.B, self.Hq, self.Hkv, self.D
        if items not in ("auto", True, False):
            raise ValueError('items must be "auto", True or False')
        parts, bpp, _ = ops.decode_plan_info(B, Hq, max_context_len, k_cache, split_tokens)
        # one-member groups put a sequence's G query heads in one MMA's 8 columns
        self.items = items if Hq // Hkv <= 8 else False
        if items is True and self.items is False:
            raise ValueError("items mode needs at most 8 query heads per kv head")
        self.blocks_per_item, self.max_items = bpp, B * parts
        sizes = [B * 8, B * 4, B * max_blocks * 4, B * Hq * D * e, B * Hkv * D * e, B * Hkv * D * e,
                 self.max_items * 16 if self.items is not False else 0]
        self.offsets, off = [], 0
        for n in sizes:
            self.offsets.append(off)
            off += _align16(n)
        self.nbytes = self.offsets[6]  # bytes copied per step without items
        self.host = [torch.zeros(off, dtype=torch.uint8).pin_memory() for _ in range(ring)]
        self.dev = torch.zeros(off, dtype=torch.uint8, device=dev)
        # views of the part copied without items (made once: slicing costs host time per step)
        self._host_meta = [h[: self.nbytes] for h in self.host]
        self._dev_meta = self.dev[: self.nbytes]
        odt = out_dtype or dtype
        self.out = torch.empty((B, Hq, D), dtype=odt, device=dev)
        self.out_host = [torch.empty((B, Hq, D), dtype=odt).pin_memory() for _ in range(ring)]
        ws = int(L.pa_decode_workspace_size(B, Hq, max_context_len, C.byref(self.desc), split_tokens))
        if self.items is not False:
            ws = max(ws, int(L.pa_decode_segments_workspace_size(B, Hq, B, 1, parts, C.byref(self.desc))))
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.dtype, self.odt, self.ring, self.i = dtype, odt, ring, 0
        self.done = [torch.cuda.Event() for _ in range(ring)]
        self.used = [False] * ring
        base = self.dev.data_ptr()
        o = self.offsets
        P = C.c_void_p
        ptr = (lambda t: P(t.data_ptr()) if t is not None else None)
        # pa_decode_append(k_new, v_new, new_dtype, slots, q, q_dtype, k_cache, v_cache, k_scale, v_scale,
        #                  tables, max_blocks, lens, max_context_len, B, Hq, scale, out, out_dtype, desc,
        #                  workspace, workspace_bytes, split_tokens, stream)
        self._head = (P(base + o[4]), P(base + o[5]), ops._TORCH_DT[dtype], P(base + o[0]), P(base + o[3]),
                      ops._TORCH_DT[dtype], ptr(k_cache), ptr(v_cache), ptr(k_scale), ptr(v_scale),
                      P(base + o[2]), max_blocks, P(base + o[1]), max_context_len, B, Hq, C.c_float(scale),
                      ptr(self.out), ops._TORCH_DT[odt], C.byref(self.desc), ptr(self.ws), self.ws.numel(),
                      split_tokens)
        # pa_decode_append_segments: the same arguments with the one-member
        # groups and the item list after `scale`; n_items (index 21) per step
        self.group_start_host = torch.arange(B + 1, dtype=torch.int32)
        self.group_start = self.group_start_host.to(dev)
        h = self._head
        self._seg_head = h[:17] + (P(self.group_start.data_ptr()), B, 1, P(base + o[6]), 0, parts) + h[17:22]
        self._split, self._hq, self._max_len = split_tokens, Hq, max_context_len
        self._n_items, self._use = C.c_int32(), C.c_int32()
        self.last_items = None  # items of the last launch (None: the fixed grid)
        self.last_copy_bytes = self.nbytes  # host-to-device bytes of the last launch
        self._keep = (k_cache, v_cache, k_scale, v_scale)
        self._L = L

    def _wait_slot(self):
        if self.used[self.i]:
            self.done[self.i].synchronize()

    def meta_ptrs(self):
        """(slots, lens, tables) ctypes pointers into the current host buffer."""
        self._wait_slot()
        base = self.host[self.i].data_ptr()
        o = self.offsets
        return (C.cast(base + o[0], C.POINTER(C.c_int64)), C.cast(base + o[1], C.POINTER(C.c_int32)),
                C.cast(base + o[2], C.POINTER(C.c_int32)))

    def inputs(self, slot=None):
        """(q, k_new, v_new) host tensors viewing the current host buffer (or
        ring slot `slot`, e.g. to fill every slot ahead)."""
        if slot is None:
            self._wait_slot()
        h, o = self.host[self.i if slot is None else slot], self.offsets
        B, Hq, Hkv, D = self.B, self.Hq, self.Hkv, self.D
        e = torch.empty((), dtype=self.dtype).element_size()
        q = h[o[3]: o[3] + B * Hq * D * e].view(self.dtype).view(B, Hq, D)
        k = h[o[4]: o[4] + B * Hkv * D * e].view(self.dtype).view(B, Hkv, D)
        v = h[o[5]: o[5] + B * Hkv * D * e].view(self.dtype).view(B, Hkv, D)
        return q, k, v

    def launch(self, stream=None):
        """Enqueue the current host buffer's step (copy in, decode, copy the
        output back) and move to the next ring slot, which the caller may
        fill while the device works; returns a handle for wait()."""
        stream = stream or torch.cuda.current_stream()
        i, L, o = self.i, self._L, self.offsets
        n_copy, n_items = self.nbytes, None
        if self.items is not False:
            base = self.host[i].data_ptr()
            use = True
            if self.items == "auto":
                ops._check(L.pa_decode_items_plan(C.c_void_p(base + o[1]), self.B, self._hq, self._max_len,
                                                  C.byref(self.desc), self._split, C.byref(self._use), None, None),
                           "pa_decode_items_plan")
                use = bool(self._use.value)
            if use:
                ops._check(L.pa_table_segments(C.c_void_p(base + o[2]), self.max_blocks, C.c_void_p(base + o[1]),
                                               C.c_void_p(self.group_start_host.data_ptr()), self.B,
                                               self.blocks_per_item, C.c_void_p(base + o[6]), self.max_items,
                                               C.byref(self._n_items), None), "pa_table_segments")
                n_items = self._n_items.value
                n_copy = o[6] + n_items * 16
        self.last_items, self.last_copy_bytes = n_items, n_copy
        with torch.cuda.stream(stream):
            if n_items is None:
                self._dev_meta.copy_(self._host_meta[i], non_blocking=True)
            else:
                self.dev[:n_copy].copy_(self.host[i][:n_copy], non_blocking=True)
            sp = C.c_void_p(stream.cuda_stream)
            if n_items is None:
                ops._check(L.pa_decode_append(*self._head, sp), "pa_decode_append")
            else:
                a = self._seg_head
                ops._check(L.pa_decode_append_segments(*a[:21], n_items, *a[22:], sp), "pa_decode_append_segments")
            self.out_host[i].copy_(self.out, non_blocking=True)
            self.done[i].record(stream)
        self.used[i] = True
        self.i = (i + 1) % self.ring
        return i

    def wait(self, handle):
        """The pinned host output [B, Hq, D] of a launched step, once ready."""
        self.done[handle].synchronize()
        return self.out_host[handle]

    def step(self, stream=None):
        """launch() and wait(): the output of the current host buffer's step."""
        return self.wait(self.launch(stream))
