#!/usr/bin/env python
"""Paged decode attention benchmark on GB300.

One step = one pass of the whole decode hot path over one batch:
  host block manager appends this step's slot for every sequence and builds
  the block tables (one pinned host->device copy), pa_cache_write stores the
  new token's K/V, pa_decode computes attention over the paged context
  (split-K partitions + merge).  The shared-prefix workload adds beam
  reselection (fork / release) and the pa_copy_blocks copy-on-write step.

Metric: KV-read GB/s of algorithmic bytes (K+V of every context token once,
plus Q, output, table entries and lengths, plus the cache-write and block-copy
bytes) per second of device time, and decode tokens/s (one token per
sequence per step).  Sequences grow by one token per step; every 64 steps the
batch is released and re-admitted at its starting lengths (as continuous
batching does when requests finish), so the workload stays the stated one.

`python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]`
prints one JSON line on rank 0.  `--impl reference` times the float64 CPU
oracle on host cores instead (bounded sample per step).
"""
import argparse
import ctypes as C
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

RESET_EVERY = 64
RING = 4              # pinned staging buffers in flight
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
METRIC = "paged decode attention KV-read GB/s and tokens/s; % of GB300 HBM peak"
METRIC_PREFILL = "multi-token paged attention KV-read GB/s and query tokens/s; % of GB300 HBM peak"
PREFILL_CONFIGS = ("prefill_mix_llama7b", "prefill_mix_llama7b_fp8", "spec_verify_gqa70b")
SERVING_CONFIGS = ("serving_llama7b",)
METRIC_SERVING = "continuous-batching serving iterations: tokens/s through scheduler + swap + cache write + attention"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1,
                   help="GPUs of the job (N > 1: launch one process per GPU with torch.distributed.run)")
    p.add_argument("--steps", type=int, default=3000, help="timed steps")
    p.add_argument("--warmup", type=int, default=50, help="untimed warm-up steps before them")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours",
                   help="reference: the float64 oracle on the host cores, bounded samples per step")
    p.add_argument("--config", default="llama7b_b32",
                   choices=["tiny", "llama7b_b32", "gqa70b_b64", "longctx_b8_f16", "longctx_b8_fp8", "longctx_b8_int8",
                            "shared_prefix_16x4"] + list(PREFILL_CONFIGS) + list(SERVING_CONFIGS),
                   help="workload: decode batches (default llama7b_b32), beam search over shared prompts, "
                        "multi-token attention mixes, or continuous-batching serving iterations")
    p.add_argument("--split", type=int, default=0, help="split_tokens (0 = library choice)")
    p.add_argument("--e2e-steps", type=int, default=300,
                   help="steps of the end-to-end measurement (host buffers in and out, waited per step)")
    p.add_argument("--unfused", action="store_true",
                   help="pa_cache_write + pa_decode instead of the fused pa_decode_append")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the oracle on the host cores")
    p.add_argument("--prefix-groups", action="store_true",
                   help="shared_prefix_16x4: pa_decode_append_grouped (each group's common prefix read once) "
                        "instead of pa_decode_append_segments (every shared block read once)")
    p.add_argument("--ungrouped", action="store_true",
                   help="shared_prefix_16x4: read shared prompt blocks once per beam (pa_decode_append)")
    p.add_argument("--fixed-grid", action="store_true",
                   help="decode batches: always pa_decode_append's fixed grid, never the host-planned list of "
                        "live partitions that pa_decode_items_plan picks for skewed lengths")
    p.add_argument("--headline-only", action="store_true",
                   help="time only --config (by default every decode workload runs and appears under `workloads`)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="wall-clock budget of the oracle baseline sample")
    return p.parse_args(argv)


# ---- multi-process plumbing (replicas only: no data-path collective) ----------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(local_seconds, local_units, world):
    """Max of the ranks' timed seconds and sum of their units (replicas)."""
    if world <= 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- measured peaks, profile traffic, clocks -----------------------------------
def _number(v):
    """A positive float from a number or from a {"value": number} / {"median": number} record."""
    if isinstance(v, dict):
        for k in ("value", "median", "gbs", "mean"):
            if k in v:
                return _number(v[k])
        return None
    try:
        x = float(v)
    except (TypeError, ValueError):
        return None
    return x if x > 0 else None


def hbm_peak():
    """The measured HBM copy bandwidth (GB/s) from MEASURED_PEAKS.json, else
    the fallback; a file in an unexpected shape falls back too."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if isinstance(d, dict):
            for key in ("hbm_gbs", "hbm_copy_gbs", "hbm_GBps"):
                x = _number(d.get(key))
                if x:
                    return x, "measured"
            for v in d.values():
                if isinstance(v, dict):
                    x = _number(v.get("hbm_gbs"))
                    if x:
                        return x, "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "device_common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_191_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(config, api):
    """DRAM bytes per decode launch from the committed ncu summary, or None
    when the kernel source changed since the counters were taken or the
    record is of another entry point (`api`, launch_api())."""
    path = os.path.join(ROOT, "profiles", f"traffic_decode_{config}.txt")
    try:
        kv = dict(line.split(":", 1) for line in open(path) if ":" in line)
    except OSError:
        return None
    if kv.get("kernel_source_sha256_16", "").strip() != kernel_source_hash():
        return None
    if kv.get("api", "").strip() != api:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples over the whole run; summaries are
    taken over the wall-clock windows in which the measured launches ran."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, index):
        self.proc = None
        self.lines = []
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]
        self.proc = None

    def rows(self):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except (ValueError, IndexError):
                continue
        return rows

    def summary(self, windows, label="timed region"):
        """Median SM clock, max clock and active throttle reasons over the
        samples that fall inside any (t0, t1) wall-clock window."""
        rows = self.rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no nvidia-smi samples"}
        inside = [r for r in rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": f"no sample inside the {label} ({len(rows)} samples in the run)"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": label}


# ---- thin CUDA driver access for the timed loop (copies and events) --------------
class Driver:
    """cuMemcpyHtoDAsync / cuEvent* through ctypes: a few microseconds less host
    time per step than the equivalent torch calls, so the loop stays ahead of
    the GPU."""

    def __init__(self):
        cu = C.CDLL("libcuda.so.1")
        cu.cuMemcpyHtoDAsync_v2.argtypes = [C.c_uint64, C.c_void_p, C.c_size_t, C.c_void_p]
        cu.cuEventCreate.argtypes = [C.POINTER(C.c_void_p), C.c_uint]
        cu.cuEventRecord.argtypes = [C.c_void_p, C.c_void_p]
        cu.cuEventSynchronize.argtypes = [C.c_void_p]
        cu.cuEventElapsedTime.argtypes = [C.POINTER(C.c_float), C.c_void_p, C.c_void_p]
        cu.cuStreamWaitEvent.argtypes = [C.c_void_p, C.c_void_p, C.c_uint]
        self.cu = cu

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed with CUresult {rc}")

    def event(self, timing=False):
        ev = C.c_void_p()
        self._ok(self.cu.cuEventCreate(C.byref(ev), 0 if timing else 2), "cuEventCreate")
        return ev

    def record(self, ev, stream):
        self._ok(self.cu.cuEventRecord(ev, stream), "cuEventRecord")

    def sync(self, ev):
        self._ok(self.cu.cuEventSynchronize(ev), "cuEventSynchronize")

    def elapsed_ms(self, a, b):
        ms = C.c_float()
        self._ok(self.cu.cuEventElapsedTime(C.byref(ms), a, b), "cuEventElapsedTime")
        return ms.value

    def wait(self, stream, ev):
        self._ok(self.cu.cuStreamWaitEvent(stream, ev, 0), "cuStreamWaitEvent")

    def h2d(self, dst_ptr, src_ptr, nbytes, stream):
        self._ok(self.cu.cuMemcpyHtoDAsync_v2(dst_ptr, src_ptr, nbytes, stream), "cuMemcpyHtoDAsync")


# ---- workloads ------------------------------------------------------------------
def load_workload(name):
    from paged_kv_cache_191_gb300 import workloads as W
    if name == "shared_prefix_16x4":
        return W.config_shared_prefix()
    return W.CONFIGS[name]()


def decode_bytes(lens, Hq, Hkv, D, kv_e, q_e, out_e):
    """Algorithmic bytes of one decode launch (K+V once, Q, out, tables, lens)."""
    lens = np.asarray(lens, dtype=np.int64)
    kv = int(lens.sum()) * Hkv * D * 2 * kv_e
    scales = int(lens.sum()) * 2 * 4 if kv_e == 1 else 0
    B = len(lens)
    tables = int(((lens + 15) // 16).sum()) * 4 + B * 4
    return kv + scales + B * Hq * D * (q_e + out_e) + tables


class DecodeStep:
    """Device-side state and the per-step host logic for a decode workload."""

    def __init__(self, w, split_tokens, steps_total, device):
        import torch
        from paged_kv_cache_191_gb300 import ops
        self.torch, self.ops, self.L = torch, ops, ops.lib()
        self.w = w
        self.B, self.Hq, self.Hkv, self.D = w.B, w.Hq, w.Hkv, w.D
        self.fp8 = w.kv_dtype in ("fp8", "int8")  # 1-byte codes + per-token scales
        self.dev = device
        self.lens0 = np.asarray(w.context_lens, dtype=np.int64)
        # capacity: lengths grow by at most RESET_EVERY tokens before a reset
        self.max_len = int(self.lens0.max()) + RESET_EVERY + 1
        self.cap = -(-self.max_len // 16)
        grow_blocks = self.B * (RESET_EVERY // 16 + 2)
        self.num_blocks = w.num_blocks + grow_blocks
        rng = np.random.Generator(np.random.PCG64(12345))
        order = np.concatenate([w.free_order, w.num_blocks + rng.permutation(grow_blocks)])
        self.order = order
        self.alloc = ops.BlockAllocator(self.num_blocks, order)
        self.ids = list(range(self.B))
        self._admit()

        kvdt = torch.float16 if w.kv_dtype in ("f16", "fp8", "int8") else torch.bfloat16
        extra = torch.zeros((grow_blocks, self.Hkv, 16, self.D), dtype=kvdt)
        kp = torch.cat([w.k_pool, extra]).to(device)
        vp = torch.cat([w.v_pool, extra]).to(device)
        if self.fp8:  # the cache is filled by the quantiser (set-up, not timed)
            N = self.num_blocks
            code_dt = torch.int8 if w.kv_dtype == "int8" else torch.uint8
            self.kc = torch.empty((N, self.Hkv, 16, self.D), dtype=code_dt, device=device)
            self.vc = torch.empty_like(self.kc)
            self.ks = torch.empty((N, 16), dtype=torch.float32, device=device)
            self.vs = torch.empty_like(self.ks)
            kin = kp.permute(0, 2, 1, 3).reshape(N * 16, self.Hkv, self.D).contiguous()
            vin = vp.permute(0, 2, 1, 3).reshape(N * 16, self.Hkv, self.D).contiguous()
            ops.cache_write(kin, vin, torch.arange(N * 16, device=device), self.kc, self.vc, self.ks, self.vs)
            del kin, vin, kp, vp
        else:
            self.kc, self.vc, self.ks, self.vs = kp, vp, None, None
        self.q = w.q.to(device)
        self.new_k, self.new_v = w.new_k.to(device), w.new_v.to(device)
        self.out = torch.empty((self.B, self.Hq, self.D), dtype=w.q.dtype, device=device)
        self.desc = ops.cache_desc(self.kc)
        self.ws_bytes = ops.decode_workspace_size(self.B, self.Hq, self.max_len, self.kc, split_tokens)
        # Items mode (set by build_step when pa_decode_items_plan picks it for
        # the batch's starting lengths): each step lists the sequences' live
        # partitions on the host (pa_table_segments over B one-member groups)
        # and runs pa_decode_append_segments instead of the fixed grid.
        self.items = False
        self.items_plan = ops.decode_items_plan(self.lens0, self.Hq, self.max_len, self.kc, split_tokens)
        _, self.blocks_per_item, self.items_per_seq = self.items_plan
        sws = int(self.L.pa_decode_segments_workspace_size(self.B, self.Hq, self.B, 1, self.items_per_seq,
                                                           C.byref(self.desc)))
        self.ws = torch.empty(max(self.ws_bytes, sws, 16), dtype=torch.uint8, device=device)
        self.split = split_tokens
        self.group_start_host = np.arange(self.B + 1, dtype=np.int32)
        self.group_start = torch.from_numpy(self.group_start_host).to(device)

        # one pinned meta buffer per ring slot: slots int64[B] | lens int32[B] | tables int32[B, cap]
        #   | items int32[B * items_per_seq][4] (16-byte aligned; items mode); a step copies the part it uses
        self.it_off = (self.B * 8 + self.B * 4 + self.B * self.cap * 4 + 15) // 16 * 16
        self.max_items = self.B * self.items_per_seq
        self.meta_bytes = self.it_off + self.max_items * 16
        self.copy_bytes = self.it_off
        self.n_items, self.n_items_c = 0, C.c_int32()
        self.meta_host = [torch.empty(self.meta_bytes, dtype=torch.uint8).pin_memory()
                          for _ in range(RING)]
        # two device copies of the meta buffer: step i+1's upload (on a copy
        # stream) overlaps step i's kernels
        self.meta_devs = [torch.empty(self.meta_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
        self.use_meta(0)
        self.drv = Driver()
        self.ring_ev = [self.drv.event() for _ in range(RING)]
        self.ring_used = [False] * RING
        self.ring = 0
        self.ids_c = (C.c_uint64 * self.B)(*self.ids)
        self.pairs_c = (C.c_int64 * (2 * self.B))()
        self.ncow = C.c_int32()
        self.cur_lens = self.lens0.copy() - 1
        self.steps_since_reset = 0
        self.blocked_s = 0.0

    def use_meta(self, i):
        self.meta_dev = self.meta_devs[i]
        self.slots_dev = self.meta_dev[: self.B * 8].view(self.torch.int64)
        self.lens_dev = self.meta_dev[self.B * 8: self.B * 12].view(self.torch.int32)
        self.tables_dev = self.meta_dev[self.B * 12: self.B * 12 + self.B * self.cap * 4].view(
            self.torch.int32).view(self.B, self.cap)

    def _admit(self):
        for b in self.ids:
            self.alloc.alloc_seq(b, int(self.w.context_lens[b]) - 1)

    def host_prepare(self, ptrs=None):
        """a1: reset if due, append one slot per sequence, tables -> pinned
        (this step's ring buffer, or the (slots, lens, tables) pointers given)."""
        ops = self.ops
        if self.steps_since_reset == RESET_EVERY:
            for b in self.ids:
                self.alloc.free_seq(b)
            self._admit()
            self.cur_lens = self.lens0.copy() - 1
            self.steps_since_reset = 0
        if ptrs is not None:
            buf = None
            slots_p, lens_p, tab_p = ptrs
        else:
            buf = self.meta_host[self.ring]
            if self.ring_used[self.ring]:
                t0 = time.perf_counter()
                self.drv.sync(self.ring_ev[self.ring])
                self.blocked_s += time.perf_counter() - t0
            base = buf.data_ptr()
            slots_p = C.cast(base, C.POINTER(C.c_int64))
            lens_p = C.cast(base + self.B * 8, C.POINTER(C.c_int32))
            tab_p = C.cast(base + self.B * 12, C.POINTER(C.c_int32))
        ops._check(self.L.pa_append_slots(self.alloc._h, self.ids_c, self.B, slots_p, self.pairs_c,
                                          C.byref(self.ncow)), "pa_append_slots")
        ops._check(self.L.pa_block_tables(self.alloc._h, self.ids_c, self.B, tab_p, self.cap, lens_p),
                   "pa_block_tables")
        if self.items and buf is not None:
            ops._check(self.L.pa_table_segments(C.c_void_p(base + self.B * 12), self.cap, C.c_void_p(base + self.B * 8),
                                                self.group_start_host.ctypes.data_as(C.c_void_p), self.B,
                                                self.blocks_per_item, C.c_void_p(base + self.it_off),
                                                self.max_items, C.byref(self.n_items_c), None),
                       "pa_table_segments")
            self.n_items = self.n_items_c.value
            self.copy_bytes = self.it_off + self.n_items * 16
        self.cur_lens += 1
        self.steps_since_reset += 1
        return buf

    def prebuild(self, stream):
        """ctypes argument tuples of this step's C calls, per device meta buffer."""
        ops, fp8 = self.ops, self.fp8
        sp = C.c_void_p(stream.cuda_stream)
        self.copy_stream = self.torch.cuda.Stream(device=self.dev)
        self.cp = C.c_void_p(self.copy_stream.cuda_stream)
        ks = C.c_void_p(self.ks.data_ptr()) if fp8 else None
        vs = C.c_void_p(self.vs.data_ptr()) if fp8 else None
        self.sp = sp
        self.write_args, self.decode_args, self.append_args = [], [], []
        for i in range(2):
            self.use_meta(i)
            self.write_args.append((C.c_void_p(self.new_k.data_ptr()), C.c_void_p(self.new_v.data_ptr()),
                                    ops._TORCH_DT[self.new_k.dtype], C.c_void_p(self.slots_dev.data_ptr()),
                                    self.B, C.c_void_p(self.kc.data_ptr()), C.c_void_p(self.vc.data_ptr()),
                                    ks, vs, C.byref(self.desc), sp))
            self.decode_args.append((C.c_void_p(self.q.data_ptr()), ops._TORCH_DT[self.q.dtype],
                                     C.c_void_p(self.kc.data_ptr()), C.c_void_p(self.vc.data_ptr()), ks, vs,
                                     C.c_void_p(self.tables_dev.data_ptr()), self.cap,
                                     C.c_void_p(self.lens_dev.data_ptr()), self.max_len, self.B, self.Hq,
                                     C.c_float(self.w.scale), C.c_void_p(self.out.data_ptr()),
                                     ops._TORCH_DT[self.out.dtype], C.byref(self.desc),
                                     C.c_void_p(self.ws.data_ptr()), self.ws.numel(), self.split, sp))
            wa, da = self.write_args[-1], self.decode_args[-1]
            # pa_decode_append(k_new, v_new, new_dtype, slot_mapping, <pa_decode args but workspace...>)
            self.append_args.append((wa[0], wa[1], wa[2], wa[3]) + da)
        # pa_decode_append_segments over one-member groups: no split_tokens;
        # n_items (index 21) is set per step
        if self.items:
            self.item_args = [a[:17] + (C.c_void_p(self.group_start.data_ptr()), self.B, 1,
                                        C.c_void_p(self.meta_devs[i].data_ptr() + self.it_off), 0,
                                        self.items_per_seq) + a[17:22] + a[23:] for i, a in enumerate(self.append_args)]
        self.use_meta(0)
        self.dbuf = 0
        self.copy_done = [self.drv.event() for _ in range(2)]
        self.used_done = [self.drv.event() for _ in range(2)]
        self.used_rec = [False, False]

    def enqueue(self, buf, ev_pair=None):
        """a1 H2D (copy stream), a2 cache write, a4+a5 decode (compute stream)."""
        L, drv, sp, cp, i = self.L, self.drv, self.sp, self.cp, self.dbuf
        if self.used_rec[i]:            # the kernels that read this device buffer are done
            drv.wait(cp, self.used_done[i])
        drv.h2d(self.meta_devs[i].data_ptr(), buf.data_ptr(), self.copy_bytes, cp)
        drv.record(self.ring_ev[self.ring], cp)
        drv.record(self.copy_done[i], cp)
        self.ring_used[self.ring] = True
        self.ring = (self.ring + 1) % RING
        drv.wait(sp, self.copy_done[i])
        if self.fused and self.items:
            a = self.item_args[i]
            self.last_item_args = a[:21] + (self.n_items,) + a[22:]  # built before the start event
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode_append_segments(*self.last_item_args)
            if st:
                self.ops._check(st, "pa_decode_append_segments")
        elif self.fused:
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode_append(*self.append_args[i])
            if st:
                self.ops._check(st, "pa_decode_append")
        else:
            st = L.pa_cache_write(*self.write_args[i])
            if st:
                self.ops._check(st, "pa_cache_write")
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode(*self.decode_args[i])
            if st:
                self.ops._check(st, "pa_decode")
        if ev_pair is not None:
            drv.record(ev_pair[1], sp)
        drv.record(self.used_done[i], sp)
        self.used_rec[i] = True
        self.dbuf ^= 1

    def _bytes_of(self, lens):
        e = 1 if self.fp8 else 2
        qe = self.q.element_size()
        dec = decode_bytes(lens, self.Hq, self.Hkv, self.D, e, qe, qe)
        write = 2 * self.B * self.Hkv * self.D * (qe + e) + (2 * self.B * 4 if self.fp8 else 0) + self.B * 8
        # the timed launch is decode plus, when fused, the cache write
        return dec + (write if self.fused else 0), dec + write + self.it_off

    def step_bytes(self, items=True):
        """(decode bytes, whole-step bytes) of the step just prepared (items
        mode: plus the item list the launch reads and the step copies)."""
        k = self.steps_since_reset  # 1..RESET_EVERY: lengths are lens0 - 1 + k
        if not hasattr(self, "_bytes_table"):
            self._bytes_table = [self._bytes_of(self.lens0 - 1 + j) for j in range(RESET_EVERY + 1)]
        d, s = self._bytes_table[k]
        if self.items and items:
            d, s = d + 16 * self.n_items, s + self.copy_bytes - self.it_off
        return d, s

    def launches_per_step(self):
        """Kernels one step launches: the decode call's own count (main kernel,
        plus the merge kernel when the library plans one) and the separate
        cache write when the write is not fused; the grouped and segment
        calls always follow their main kernel with their merge kernel."""
        if (getattr(self, "grouped", False) or self.items) and self.fused:
            return 2
        _, _, kernels = self.ops.decode_plan_info(self.B, self.Hq, self.max_len, self.kc, self.split)
        return kernels + (0 if self.fused else 1)


class SharedPrefixStep(DecodeStep):
    """Beam search over shared prompts: every step each group's beams are
    reselected from parent beams (fork all children, then release the old
    beams), one slot is appended per beam -- copy-on-write where siblings
    share a partially filled block -- and pa_copy_blocks runs before the
    cache write and the decode."""

    def __init__(self, w, split_tokens, steps_total, device):
        import torch
        from paged_kv_cache_191_gb300 import ops
        self.torch, self.ops, self.L = torch, ops, ops.lib()
        self.w = w
        self.B, self.Hq, self.Hkv, self.D = w.B, w.Hq, w.Hkv, w.D
        self.fp8 = False
        self.items = False  # the groups' segment items instead (below)
        self.dev = device
        self.alloc = ops.BlockAllocator(w.num_blocks, w.free_order)
        self.roots = [10 ** 9 + g for g in range(w.groups)]
        for r in self.roots:
            self.alloc.alloc_seq(r, w.prompt_len)
        self.next_id = 0
        self._admit()
        self.max_len = w.prompt_len + int(w.tail_lens.max()) + RESET_EVERY + 1
        self.cap = -(-self.max_len // 16)
        self.kc, self.vc = w.k_pool.to(device), w.v_pool.to(device)
        self.ks = self.vs = None
        # the step's model inputs (q, k_new, v_new) packed in one device buffer,
        # so the end-to-end run moves them with one copy
        nq, nkv = self.B * self.Hq * self.D, self.B * self.Hkv * self.D
        self.qkv = torch.empty(nq + 2 * nkv, dtype=w.q.dtype, device=device)
        self.q = self.qkv[:nq].view(self.B, self.Hq, self.D)
        self.new_k = self.qkv[nq: nq + nkv].view(self.B, self.Hkv, self.D)
        self.new_v = self.qkv[nq + nkv:].view(self.B, self.Hkv, self.D)
        self.q.copy_(w.q)
        self.new_k.copy_(w.new_k)
        self.new_v.copy_(w.new_v)
        self.out = torch.empty((self.B, self.Hq, self.D), dtype=w.q.dtype, device=device)
        self.desc = ops.cache_desc(self.kc)
        self.ws_bytes = ops.decode_workspace_size(self.B, self.Hq, self.max_len, self.kc, split_tokens)
        # groups: the beams of one prompt.  Segments (default): the runs of
        # table positions each subset of a group's beams holds (the prompt,
        # blocks inherited from a parent, private tails), every block read
        # once; prefix groups: each group's longest common run of leading
        # table entries read once, the rest per beam.  Either is computed per
        # step from the block manager's tables and staged with the metadata.
        self.grouped = True
        self.segments = True
        self.group_start_host = np.arange(0, self.B + 1, w.beams, dtype=np.int32)
        self.group_start = torch.from_numpy(self.group_start_host).to(device)
        self.max_group_items = 32   # items per group: ~7 segments of <= 40 blocks for 4 beams
        self.blocks_per_item = 40   # item lengths 16 / 24 / 32 / 40 / 48 / 56 / 64 measured 71.6 / 73.2 / 69.5 / 64.9 / 65.2 / 66.2 / 67.3 us
        gws = int(self.L.pa_decode_grouped_workspace_size(self.B, self.Hq, self.max_len, w.groups, w.beams,
                                                          self.cap, C.byref(self.desc), split_tokens))
        sws = int(self.L.pa_decode_segments_workspace_size(self.B, self.Hq, w.groups, w.beams,
                                                           self.max_group_items, C.byref(self.desc)))
        self.ws = torch.empty(max(self.ws_bytes, gws, sws, 16), dtype=torch.uint8, device=device)
        self.split = split_tokens
        # meta: slots int64[B] | pairs int64[B, 2] | lens int32[B] | tables int32[B, cap] | prefix int32[groups]
        #       | items int32[max_items][4] (16-byte aligned); a step copies the part it uses
        self.pre_off = self.B * 8 + self.B * 16 + self.B * 4 + self.B * self.cap * 4
        self.it_off = (self.pre_off + w.groups * 4 + 15) // 16 * 16
        self.max_items = w.groups * self.max_group_items
        self.most_c = C.c_int32()
        self.meta_bytes = self.it_off + self.max_items * 16
        self.copy_bytes = self.pre_off + w.groups * 4
        self.n_items = 0
        self.n_items_c = C.c_int32()
        self.meta_host = [torch.empty(self.meta_bytes, dtype=torch.uint8).pin_memory() for _ in range(RING)]
        self.meta_devs = [torch.empty(self.meta_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
        self.use_meta(0)
        self.drv = Driver()
        self.ring_ev = [self.drv.event() for _ in range(RING)]
        self.ring_used = [False] * RING
        self.ring = 0
        self.ncow_c = C.c_int32()
        self.blocked_s = 0.0
        self.steps_since_reset = 0
        self.step_idx = 0
        self.lens0 = np.full(self.B, w.prompt_len) + w.tail_lens.reshape(-1)
        self.cur_lens = self.lens0.copy()
        self.history = []  # per timed step: (tables, lens, n_cow) for the byte count

    def use_meta(self, i):
        T = self.torch
        self.meta_dev = self.meta_devs[i]
        B = self.B
        self.slots_dev = self.meta_dev[: B * 8].view(T.int64)
        self.pairs_dev = self.meta_dev[B * 8: B * 24].view(T.int64).view(B, 2)
        self.lens_dev = self.meta_dev[B * 24: B * 28].view(T.int32)
        self.tables_dev = self.meta_dev[B * 28: self.pre_off].view(T.int32).view(B, self.cap)
        self.prefix_dev = self.meta_dev[self.pre_off: self.pre_off + self.w.groups * 4].view(T.int32)

    def prebuild(self, stream):
        super().prebuild(stream)
        w = self.w
        # pa_decode_append's arguments with the group description after `scale`
        self.grouped_args, self.segment_args = [], []
        for i, a in enumerate(self.append_args):
            pre = C.c_void_p(self.meta_devs[i].data_ptr() + self.pre_off)
            extra = (C.c_void_p(self.group_start.data_ptr()), pre, w.groups, w.beams, self.cap)
            self.grouped_args.append(a[:17] + extra + a[17:])
            # pa_decode_append_segments: no split_tokens; n_items (index 21) is set per step
            seg = (C.c_void_p(self.group_start.data_ptr()), w.groups, w.beams,
                   C.c_void_p(self.meta_devs[i].data_ptr() + self.it_off), 0, self.max_group_items)
            self.segment_args.append(a[:17] + seg + a[17:22] + a[23:])

    def seg_call_args(self, i):
        a = self.segment_args[i]
        return a[:21] + (self.n_items,) + a[22:]

    def stage_segments(self, base):
        """Each group's segment items (pa_table_segments) from the tables and
        lengths the block manager just staged in the pinned metadata buffer at
        `base`, written beside them."""
        B, w = self.B, self.w
        st = self.L.pa_table_segments(C.c_void_p(base + B * 28), self.cap, C.c_void_p(base + B * 24),
                                      self.group_start_host.ctypes.data_as(C.c_void_p), w.groups,
                                      self.blocks_per_item, C.c_void_p(base + self.it_off), self.max_items,
                                      C.byref(self.n_items_c), C.byref(self.most_c))
        if st:
            self.ops._check(st, "pa_table_segments")
        self.n_items = self.n_items_c.value
        if self.most_c.value > self.max_group_items:
            raise RuntimeError("a group needs more than max_group_items segment items")
        self.copy_bytes = self.it_off + self.n_items * 16

    def stage_prefix(self, raw):
        """Each group's shared prefix (ops.shared_table_prefix) from the tables
        and lengths the block manager just staged in `raw`, the pinned
        metadata buffer, written beside them."""
        w, B = self.w, self.B
        tables = raw[B * 28: self.pre_off].view(np.int32).reshape(B, self.cap)
        lens = raw[B * 24: B * 28].view(np.int32)
        self.ops.shared_table_prefix(tables, lens, self.group_start_host,
                                     out=raw[self.pre_off: self.pre_off + w.groups * 4].view(np.int32))

    def _fresh(self, n):
        ids = np.arange(self.next_id, self.next_id + n, dtype=np.uint64)
        self.next_id += n
        return ids

    def _admit(self):
        """Beams forked from their group's prompt, grown by their tails."""
        w = self.w
        self.ids = self._fresh(self.B)
        self.ids_c = self.ids.ctypes.data_as(C.POINTER(C.c_uint64))
        self.alloc.fork_seqs([self.roots[i // w.beams] for i in range(self.B)], [int(x) for x in self.ids])
        for i, sid in enumerate(self.ids):
            _, cow = self.alloc.append_tokens(int(sid), int(w.tail_lens.reshape(-1)[i]), want_slots=False)
            assert cow[0] < 0  # the 1024-token prompt fills its last block
        # parent row of every new beam, per reselection pattern
        if not hasattr(self, "par_rows"):
            g = np.arange(w.groups)[:, None] * w.beams
            self.par_rows = [(g + w.parents[k]).reshape(-1).astype(np.int32) for k in range(len(w.parents))]

    def host_prepare(self):
        w, B = self.w, self.B
        if self.steps_since_reset == RESET_EVERY:
            self.alloc.free_seqs([int(x) for x in self.ids])
            self._admit()
            self.cur_lens = self.lens0.copy()
            self.steps_since_reset = 0
        # beam reselection: beam i continues from beam par[i] of its group
        par = self.par_rows[self.step_idx % len(self.par_rows)]
        self.ops._check(self.L.pa_reselect(self.alloc._h, self.ids_c, par.ctypes.data_as(C.POINTER(C.c_int32)), B),
                        "pa_reselect")
        buf = self.meta_host[self.ring]
        if self.ring_used[self.ring]:
            t0 = time.perf_counter()
            self.drv.sync(self.ring_ev[self.ring])
            self.blocked_s += time.perf_counter() - t0
        base = buf.data_ptr()
        self.ops._check(self.L.pa_append_slots(self.alloc._h, self.ids_c, B, C.cast(base, C.POINTER(C.c_int64)),
                                               C.cast(base + B * 8, C.POINTER(C.c_int64)), C.byref(self.ncow_c)),
                        "pa_append_slots")
        self.ops._check(self.L.pa_block_tables(self.alloc._h, self.ids_c, B, C.cast(base + B * 28, C.POINTER(C.c_int32)),
                                               self.cap, C.cast(base + B * 24, C.POINTER(C.c_int32))),
                        "pa_block_tables")
        if self.grouped and self.segments:
            self.stage_segments(base)
        else:
            self.stage_prefix(buf.numpy())
            self.copy_bytes = self.pre_off + w.groups * 4
        self.n_cow = self.ncow_c.value
        self.steps_since_reset += 1
        self.step_idx += 1
        return buf

    def enqueue(self, buf, ev_pair=None):
        """a1 H2D (copy stream), a3 block copies, a2 cache write, a4+a5 decode."""
        L, drv, sp, cp, i = self.L, self.drv, self.sp, self.cp, self.dbuf
        if self.used_rec[i]:
            drv.wait(cp, self.used_done[i])
        drv.h2d(self.meta_devs[i].data_ptr(), buf.data_ptr(), self.copy_bytes, cp)
        drv.record(self.ring_ev[self.ring], cp)
        drv.record(self.copy_done[i], cp)
        self.ring_used[self.ring] = True
        self.ring = (self.ring + 1) % RING
        drv.wait(sp, self.copy_done[i])
        if self.n_cow:
            st = L.pa_copy_blocks(C.c_void_p(self.kc.data_ptr()), C.c_void_p(self.vc.data_ptr()), None, None,
                                  C.c_void_p(self.meta_devs[i].data_ptr() + self.B * 8), self.n_cow,
                                  C.byref(self.desc), sp)
            if st:
                self.ops._check(st, "pa_copy_blocks")
        if self.fused and self.grouped and self.segments:
            # the argument tuple is built before the start event: nothing that
            # allocates (and may run the garbage collector) sits between the
            # event and the launch
            self.last_seg_args = self.seg_call_args(i)
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode_append_segments(*self.last_seg_args)
            if st:
                self.ops._check(st, "pa_decode_append_segments")
        elif self.fused and self.grouped:
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode_append_grouped(*self.grouped_args[i])
            if st:
                self.ops._check(st, "pa_decode_append_grouped")
        elif self.fused:
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode_append(*self.append_args[i])
            if st:
                self.ops._check(st, "pa_decode_append")
        else:
            st = L.pa_cache_write(*self.write_args[i])
            if st:
                self.ops._check(st, "pa_cache_write")
            if ev_pair is not None:
                drv.record(ev_pair[0], sp)
            st = L.pa_decode(*self.decode_args[i])
            if st:
                self.ops._check(st, "pa_decode")
        if ev_pair is not None:
            drv.record(ev_pair[1], sp)
        drv.record(self.used_done[i], sp)
        self.used_rec[i] = True
        self.dbuf ^= 1

    def step_bytes(self):
        """Recorded now, counted after the timed loop (unique physical bytes)."""
        buf = self.meta_host[(self.ring - 0) % RING]
        B = self.B
        raw = buf.numpy()
        lens = raw[B * 24: B * 28].view(np.int32).copy()
        tables = raw[B * 28: self.pre_off].view(np.int32).reshape(B, self.cap).copy()
        self.history.append((tables, lens, self.n_cow))
        return 0, 0

    def as_decode_workload(self):
        """The current batch as a plain decode workload (for the CPU oracle)."""
        from types import SimpleNamespace
        tables, lens = self.alloc.tables([int(x) for x in self.ids], self.cap)
        w = self.w
        return SimpleNamespace(name=w.name, B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, kv_dtype="f16",
                               context_lens=lens, block_tables=tables, k_pool=w.k_pool, v_pool=w.v_pool,
                               q=w.q, scale=w.scale)

    def count_bytes(self, history=None):
        """(decode bytes, whole-step bytes, logical decode bytes) summed over history.

        Shared-prefix blocks count once per step (unique physical bytes); the
        logical figure counts every beam's context separately."""
        e, qe = 2, self.q.element_size()
        row = self.Hkv * self.D * 2 * e                # K+V bytes of one token
        block_bytes = self.Hkv * 16 * self.D * e
        dec_u = step_u = dec_l = 0
        j = np.arange(self.cap)[None, :]
        for tables, lens, ncow in (self.history if history is None else history):
            nb = (lens[:, None] + 15) // 16
            rows = np.where(j < nb - 1, 16, np.where(j == nb - 1, lens[:, None] - 16 * (nb - 1), 0))
            live = rows > 0
            blk, used = tables[live], rows[live]
            order = np.lexsort((-used, blk))          # per block, largest use first
            blk, used = blk[order], used[order]
            first = np.r_[True, blk[1:] != blk[:-1]]
            extra = self.B * self.Hq * self.D * 2 * qe + int(nb.sum()) * 4 + self.B * 4
            d = int(used[first].sum()) * row + extra
            dl = int(lens.sum()) * row + extra
            write = 2 * self.B * self.Hkv * self.D * 2 * e + self.B * 8
            copy = ncow * 2 * 2 * block_bytes
            dec_u += d + (write if self.fused else 0)
            dec_l += dl
            step_u += d + write + copy + self.copy_bytes
        return dec_u, step_u, dec_l


DECODE_WORKLOADS = ("llama7b_b32", "gqa70b_b64", "longctx_b8_f16", "longctx_b8_fp8", "longctx_b8_int8",
                    "shared_prefix_16x4")
CLOCK_HOLD_S = 0.6   # the sampler's period is 50 ms: hold a short timed region's load this long


def build_step(name, args, dev):
    """Device state and host logic of one decode workload."""
    w = load_workload(name)
    shared = name == "shared_prefix_16x4"
    st = (SharedPrefixStep if shared else DecodeStep)(w, args.split, args.steps + args.warmup, dev)
    st.fused = not args.unfused
    if shared:
        st.grouped = not args.ungrouped
        st.segments = not args.prefix_groups
    else:
        st.items = st.fused and st.items_plan[0] and not args.fixed_grid
    return w, st, shared


def time_steps(st, shared, stream, args, world):
    """W warm-up steps, a barrier, then exactly K steps between two events on
    the launch stream, each decode launch bracketed by its own event pair."""
    import torch
    dec_events = [(st.drv.event(True), st.drv.event(True)) for _ in range(args.steps)]
    t_start, t_end = st.drv.event(True), st.drv.event(True)
    r = {}
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            st.enqueue(st.host_prepare())
        if shared:
            st.history.clear()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        dec_b = step_b = 0
        st.blocked_s = 0.0
        # no garbage-collector pause inside the timed steps: a pause between a
        # launch's start event and its submission would count in its time
        gc_was = gc.isenabled()
        gc.disable()
        wall0 = time.time()
        st.drv.record(t_start, st.sp)
        for i in range(args.steps):
            buf = st.host_prepare()
            d, s = st.step_bytes()
            dec_b += d
            step_b += s
            st.enqueue(buf, dec_events[i])
        st.drv.record(t_end, st.sp)
        host_done = time.time()
        if gc_was:
            gc.enable()
        if shared:
            dec_b, step_b, r["dec_logical"] = st.count_bytes()
            r["copies"] = sum(h[2] for h in st.history) / args.steps
            r["cow_launches"] = sum(1 for h in st.history if h[2] > 0)  # one pa_copy_blocks per copying step
        stream.synchronize()
        wall1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    errs = st.ops.device_errors(clear=True)
    if errs:
        raise RuntimeError(f"device error flags {errs:#x} during the benchmark")
    r.update(local_s=st.drv.elapsed_ms(t_start, t_end) / 1e3,
             dec_list=[st.drv.elapsed_ms(a, b) for a, b in dec_events],
             dec_b=dec_b, step_b=step_b, wall0=wall0, wall1=wall1, host_done=host_done,
             blocked_s=st.blocked_s)
    r["dec_ms"] = sum(r["dec_list"]) / args.steps
    return r


def decode_call(st):
    """(function, arguments) of the last step's decode launch: re-issuing it
    rewrites the same slots with the same rows, so every repeat is the same work."""
    i = st.dbuf ^ 1
    if st.fused and getattr(st, "grouped", False) and isinstance(st, SharedPrefixStep):
        if st.segments:
            return st.L.pa_decode_append_segments, st.last_seg_args
        return st.L.pa_decode_append_grouped, st.grouped_args[i]
    if st.fused and st.items:
        return st.L.pa_decode_append_segments, st.last_item_args
    if st.fused:
        return st.L.pa_decode_append, st.append_args[i]
    return st.L.pa_decode, st.decode_args[i]


def clock_windows(st, stream, r):
    """Wall-clock windows in which this workload's decode launches ran: the
    timed region and, when it is shorter than CLOCK_HOLD_S, the same launch
    re-issued back to back (untimed) until it has run that long, so that the
    clock sampler sees the SM clock under this load."""
    import torch
    windows = [(r["wall0"], r["wall1"])]
    label = "timed region"
    span = r["wall1"] - r["wall0"]
    if span < CLOCK_HOLD_S:
        fn, fargs = decode_call(st)
        n = max(1, int((CLOCK_HOLD_S - span) / max(r["dec_ms"] / 1e3, 1e-6)))
        with torch.cuda.stream(stream):
            stream.synchronize()
            h0 = time.time()
            for k in range(n):
                st.ops._check(fn(*fargs), "decode")
                if k % 256 == 255:  # keep the launch queue short
                    stream.synchronize()
            stream.synchronize()
            h1 = time.time()
        windows.append((h0, h1))
        label = (f"timed region ({span * 1e3:.1f} ms) + {n} more launches of the last step's decode, "
                 f"back to back, {(h1 - h0) * 1e3:.0f} ms")
    return windows, label


def launch_api(st, shared):
    """The entry point a decode workload's timed launch goes through."""
    if shared and st.fused and st.grouped:
        return "pa_decode_append_segments" if st.segments else "pa_decode_append_grouped"
    if st.fused:
        return "pa_decode_append_segments (one-member groups)" if st.items else "pa_decode_append"
    return "pa_decode"


def launch_kernel_name(st, shared):
    if shared and st.fused and st.grouped and st.segments:
        return ("pa_decode_append_segments (decode_main over the groups' shared-block segments with the fused "
                "cache write + decode_reduce_segments)")
    if shared and st.fused and st.grouped:
        return ("pa_decode_append_grouped (decode_main over shared-prefix groups with the fused "
                "cache write + decode_reduce_grouped)")
    if st.fused and st.items:
        return ("pa_decode_append_segments over one-member groups (decode_main over the live partitions the host "
                "lists with pa_table_segments, fused cache write + decode_reduce_segments)")
    if st.fused:
        return "pa_decode_append (decode_main with the fused cache write + decode_reduce)"
    return "pa_decode (decode_main + decode_reduce)"


def workload_entry(name, w, st, shared, r, args, peak, clock):
    """One decode workload's figures for the JSON line's `workloads` table."""
    avg = r["dec_b"] / args.steps
    achieved = avg / (r["dec_ms"] / 1e3) / 1e9
    e = {"kv_dtype": w.kv_dtype, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
         "launch_ms": round(r["dec_ms"], 5), "per_launch_ms": pct(r["dec_list"]),
         "bytes_per_launch": int(avg), "kv_gbs": round(achieved, 2), "frac": round(achieved / peak, 4),
         "tokens_per_s": round(st.B / (r["dec_ms"] / 1e3), 1),
         "ms_per_step": round(r["local_s"] * 1e3 / args.steps, 5),
         "step_gbs": round(r["step_b"] / r["local_s"] / 1e9, 2),
         "gpu_launches": st.launches_per_step() * args.steps + r.get("cow_launches", 0),
         "kernel": launch_kernel_name(st, shared), "api": launch_api(st, shared),
         "traffic": profiled_traffic(name, launch_api(st, shared)), "clocks": clock}
    if shared:
        e["bytes"] = "unique physical bytes (shared blocks once per step)"
        e["logical_kv_gbs"] = round(r["dec_logical"] / args.steps / (r["dec_ms"] / 1e3) / 1e9, 2)
        e["copies_per_step"] = round(r["copies"], 2)
    return e


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    clocks = ClockSampler(local_rank)
    clocks.start()  # before set-up: the sampler's first lines take a moment to arrive
    w, st, shared = build_step(args.config, args, dev)
    stream = torch.cuda.Stream(device=dev)
    st.prebuild(stream)
    r = time_steps(st, shared, stream, args, world)
    local_s, dec_ms, dec_b, step_b = r["local_s"], r["dec_ms"], r["dec_b"], r["step_b"]
    max_s, tot_bytes = aggregate(local_s, float(step_b), world)
    _, tot_tokens = aggregate(local_s, float(st.B * args.steps), world)
    windows, label = clock_windows(st, stream, r)

    # e2e: public Python API, host (pinned) inputs in, result out, every step
    dec_list = r["dec_list"]
    timing = timing_detail(st, stream, dec_list) if not shared else {"per_launch_ms": pct(dec_list)}
    e2e = run_e2e(st, args, stream)
    swap = measure_swap(st, stream)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(st.as_decode_workload() if shared else w, args.cpu_seconds)
    peak, peak_kind = hbm_peak()
    avg_dec_bytes = dec_b / args.steps
    achieved = avg_dec_bytes / (dec_ms / 1e3) / 1e9
    traffic = profiled_traffic(args.config, launch_api(st, shared))
    head_entry = workload_entry(args.config, w, st, shared, r, args, peak, None)
    launches = head_entry["gpu_launches"]
    del st
    torch.cuda.empty_cache()

    # every other decode workload, same steps / warm-up, in the same process
    others = {}
    if not args.headline_only:
        for name in DECODE_WORKLOADS:
            if name == args.config:
                continue
            ow, ost, oshared = build_step(name, args, dev)
            ost.prebuild(stream)
            orr = time_steps(ost, oshared, stream, args, world)
            ow_windows, ow_label = clock_windows(ost, stream, orr)
            entry = workload_entry(name, ow, ost, oshared, orr, args, peak, None)
            others[name] = (entry, ow_windows, ow_label)
            launches += entry["gpu_launches"]
            del ow, ost
            torch.cuda.empty_cache()
    clocks.stop()
    all_windows = list(windows)
    head_entry["clocks"] = clocks.summary(windows, label)
    workloads = {args.config: head_entry}
    for name, (entry, ow_windows, ow_label) in others.items():
        entry["clocks"] = clocks.summary(ow_windows, ow_label)
        all_windows += ow_windows
        workloads[name] = entry
    res = {
        "metric": METRIC,
        "value": round(tot_bytes / max_s / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"f16": "f16", "bf16": "bf16", "fp8": "fp8e4m3(kv)/f16", "int8": "int8(kv)/f16"}[w.kv_dtype]
                 + "+f32acc",
        "data": "synthetic",
        "config": {
            "workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
            "block_size": 16, "kv_dtype": w.kv_dtype,
            "context_lens": f"start {int(st_lens0(w, shared).min())}..{int(st_lens0(w, shared).max())} "
                            f"(mean {st_lens0(w, shared).mean():.0f}), +1 per step, batch re-admitted every "
                            f"{RESET_EVERY} steps",
            **({"sharing": "16 groups x 4 beams share a 1024-token prompt; beams reselected from "
                           "parents every step (fork + release), copy-on-write before each decode; "
                           "bytes count shared blocks once (logical bytes reported separately)",
                "prompt_reads": ("every shared block once (pa_decode_append_segments)"
                                 if not args.unfused and not args.ungrouped and not args.prefix_groups
                                 else "once per group of 4 beams (pa_decode_append_grouped)"
                                 if not args.unfused and not args.ungrouped else "once per beam")}
               if shared else {}),
            "split_tokens": args.split or "auto",
            "l2": f"no flush: K+V per step {avg_dec_bytes / 1e6:.0f} MB vs 129 MB L2",
            "parallelism": f"replicas x{world}",
        },
        "tokens_per_s": round(tot_tokens / max_s, 1),
        **({"logical_decode_gbs": round(r["dec_logical"] / args.steps / (dec_ms / 1e3) / 1e9, 2),
            "copies_per_step": round(r["copies"], 2)} if shared else {}),
        "host_us_per_step": {"busy": round((r["host_done"] - r["wall0"] - r["blocked_s"]) * 1e6 / args.steps, 2),
                             "blocked_on_gpu": round(r["blocked_s"] * 1e6 / args.steps, 2)},
        "kv_gbs_decode_only": round(achieved, 2),
        "pct_of_nominal_8TBs": round(100 * tot_bytes / max_s / 1e9 / NOMINAL_HBM_GBS, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": traffic, "kernel": head_entry["kernel"], "api": head_entry["api"],
                     "bytes_per_launch": int(avg_dec_bytes), "launch_ms": round(dec_ms, 5)},
        "timing": timing,
        "e2e": e2e,
        "swap": swap,
        "gpu_launches": launches,
        "clocks": clocks.summary(all_windows, "timed regions of every workload in this line (and their "
                                              "clock holds)"),
        "cpu_baseline": cpu,
        "workloads": workloads,
    }
    if rank == 0:
        print(json.dumps(res), flush=True)


def st_lens0(w, shared):
    """Starting context lengths of a decode workload (shared prefix: prompt + tail)."""
    if shared:
        return np.full(w.B, w.prompt_len) + w.tail_lens.reshape(-1)
    return np.asarray(w.context_lens, dtype=np.int64)


def pct(xs):
    xs = np.asarray(xs, dtype=np.float64)
    return {"median": round(float(np.median(xs)), 5), "p10": round(float(np.percentile(xs, 10)), 5),
            "p90": round(float(np.percentile(xs, 90)), 5), "n": int(len(xs))}


def timing_detail(st, stream, dec_ms, reps=100):
    """The decode launch timed three more ways, on the last step's inputs
    (the fused write rewrites the same slots, so every rep is the same work):
    after an L2 flush (a 2 x L2 buffer written between reps, outside the
    events), back to back on the stream, and replayed from a CUDA graph."""
    torch = st.torch
    L, drv, sp = st.L, st.drv, st.sp
    fn, args = decode_call(st)
    out = {"per_launch_ms": pct(dec_ms)}
    l2 = int(getattr(torch.cuda.get_device_properties(st.dev), "L2_cache_size", 128 << 20))
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=st.dev)
    evs = [(drv.event(True), drv.event(True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        stream.synchronize()
        for a, b in evs:
            flush.zero_()
            drv.record(a, sp)
            st.ops._check(fn(*args), "decode")
            drv.record(b, sp)
        stream.synchronize()
        out["l2_flushed_ms"] = dict(pct([drv.elapsed_ms(a, b) for a, b in evs]), flush_bytes=2 * l2)
        t0, t1 = drv.event(True), drv.event(True)
        drv.record(t0, sp)
        for _ in range(reps):
            st.ops._check(fn(*args), "decode")
        drv.record(t1, sp)
        stream.synchronize()
        out["stream_ms_per_launch"] = round(drv.elapsed_ms(t0, t1) / reps, 5)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            st.ops._check(fn(*args), "decode")
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            drv.record(t0, sp)
            for _ in range(reps):
                g.replay()
            drv.record(t1, sp)
            stream.synchronize()
        out["graph_ms_per_launch"] = round(drv.elapsed_ms(t0, t1) / reps, 5)
    except Exception as e:  # reported, not fatal: the graph figure is supplementary
        out["graph_ms_per_launch"] = None
        out["graph_error"] = str(e)[:200]
    del flush
    return out


def measure_swap(st, stream, n_seqs=8, reps=5):
    """Preemption traffic: the blocks of n_seqs sequences to a pinned host pool
    and back (pa_swap_blocks, one gather launch per direction), event-timed."""
    import torch
    n_seqs = min(n_seqs, st.B)
    ids = [int(x) for x in (st.ids[:n_seqs] if hasattr(st, "ids") and not isinstance(st.ids, list)
                            else list(range(n_seqs)))]
    tables, lens = st.alloc.tables(ids, st.cap)
    blocks = [int(b) for row, n in zip(tables, lens) for b in row[: -(-int(n) // 16)]]
    nb = len(blocks)
    shape = (nb,) + tuple(st.kc.shape[1:])
    hk = torch.empty(shape, dtype=st.kc.dtype).pin_memory()
    hv = torch.empty(shape, dtype=st.kc.dtype).pin_memory()
    hks = torch.empty((nb, 16)).pin_memory() if st.fp8 else None
    hvs = torch.empty((nb, 16)).pin_memory() if st.fp8 else None
    out_pairs = torch.tensor([[b, i] for i, b in enumerate(blocks)], dtype=torch.int64, device=st.dev)
    in_pairs = torch.tensor([[i, b] for i, b in enumerate(blocks)], dtype=torch.int64, device=st.dev)
    ev = [st.drv.event(True) for _ in range(3)]
    sp = C.c_void_p(stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(2):  # warm-up
            st.ops.swap_blocks(hk, hv, st.kc, st.vc, out_pairs, hks, hvs, st.ks, st.vs, stream=stream)
            st.ops.swap_blocks(st.kc, st.vc, hk, hv, in_pairs, st.ks, st.vs, hks, hvs, stream=stream)
        st.drv.record(ev[0], sp)
        for _ in range(reps):
            st.ops.swap_blocks(hk, hv, st.kc, st.vc, out_pairs, hks, hvs, st.ks, st.vs, stream=stream)
        st.drv.record(ev[1], sp)
        for _ in range(reps):
            st.ops.swap_blocks(st.kc, st.vc, hk, hv, in_pairs, st.ks, st.vs, hks, hvs, stream=stream)
        st.drv.record(ev[2], sp)
        stream.synchronize()
    nbytes = 2 * hk[0].numel() * hk.element_size() * nb + (2 * 64 * nb if st.fp8 else 0)
    t_out = st.drv.elapsed_ms(ev[0], ev[1]) / reps / 1e3
    t_in = st.drv.elapsed_ms(ev[1], ev[2]) / reps / 1e3
    return {"sequences": len(ids), "blocks": nb, "bytes_per_direction": nbytes,
            "out_gbs": round(nbytes / t_out / 1e9, 1), "in_gbs": round(nbytes / t_in / 1e9, 1),
            "path": "GPU cache <-> pinned host pool, device-side gather (NVLink-C2C)"}


def run_e2e(st, args, stream):
    """Same step through the public API with pinned host inputs in and the
    output back, synced every step: DecodeSession (one staging copy of the
    step's q / k_new / v_new and block-manager output, one fused launch, one
    output copy) for the decode workloads; ops.* calls for the shared-prefix
    workload."""
    import torch
    ops = st.ops
    n = max(1, min(args.e2e_steps, args.steps))
    if not isinstance(st, SharedPrefixStep):
        from paged_kv_cache_191_gb300.session import DecodeSession
        sess = DecodeSession(st.kc, st.vc, st.B, st.Hq, st.cap, st.max_len, st.w.scale, st.q.dtype,
                             k_scale=st.ks, v_scale=st.vs, split_tokens=st.split,
                             items="auto" if st.items else False)
        for r in range(sess.ring):  # the model's outputs for the step (the same every step here)
            q, k, v = sess.inputs(slot=r)
            q.copy_(st.w.q)
            k.copy_(st.w.new_k)
            v.copy_(st.w.new_v)
        total_b = h2d_b = listed = 0
        with torch.cuda.stream(stream):
            stream.synchronize()
            t0 = time.perf_counter()
            st.host_prepare(sess.meta_ptrs())
            for k in range(n):
                _, s = st.step_bytes(items=False)
                h = sess.launch(stream)
                total_b += s + sess.last_copy_bytes - sess.nbytes  # the session's item list, when it lists
                h2d_b += sess.last_copy_bytes
                listed += sess.last_items is not None
                if k + 1 < n:  # the block manager prepares the next step while this one runs
                    st.host_prepare(sess.meta_ptrs())
                out = sess.wait(h)
            t1 = time.perf_counter()
        return {"value": round(total_b / (t1 - t0) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d_b // n), "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "steps": n, "tokens_per_s": round(st.B * n / (t1 - t0), 1),
                "steps_with_item_list": listed,
                "api": "paged_kv_cache_191_gb300.session.DecodeSession (block manager writes into a pinned staging "
                       "buffer beside q / k_new / v_new, the next step's while the current one runs; one H2D copy, "
                       "pa_decode_append -- or, when pa_decode_items_plan picks it for the step's lengths, the "
                       "live partitions listed by pa_table_segments and pa_decode_append_segments -- one D2H copy "
                       "of the output, waited for every step)"}
    # Shared-prefix beam search: the timed step's own path (block manager ->
    # pinned metadata with the groups' prefixes -> one copy; copy-on-write
    # copies; the grouped fused decode) plus the model's inputs from pinned
    # host memory (q, k_new, v_new packed: one copy) and the output back (one
    # copy), waited for every step.
    hqkv = torch.empty(st.qkv.shape, dtype=st.qkv.dtype).pin_memory()
    hqkv.copy_(st.qkv)
    hout = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    st.history.clear()
    drv, sp = st.drv, st.sp
    with torch.cuda.stream(stream):
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            buf = st.host_prepare()
            st.step_bytes()
            drv.h2d(st.qkv.data_ptr(), hqkv.data_ptr(), hqkv.numel() * hqkv.element_size(), sp)
            st.enqueue(buf)
            hout.copy_(st.out, non_blocking=True)
            stream.synchronize()
        t1 = time.perf_counter()
    total_b = st.count_bytes()[1]
    st.history.clear()
    h2d = st.copy_bytes + hqkv.numel() * hqkv.element_size()
    d2h = hout.numel() * hout.element_size()
    return {"value": round(total_b / (t1 - t0) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "tokens_per_s": round(st.B * n / (t1 - t0), 1),
            "api": "libpagedkv C ABI through the benchmark's step (block manager writes slots, copy pairs, tables "
                   "and the groups' segment items (pa_table_segments) into a pinned staging buffer; one H2D copy "
                   "of it and one of the packed q / k_new / v_new; pa_copy_blocks; pa_decode_append_segments; one "
                   "D2H copy of the output; waited for every step)"}


# ---- multi-token workloads (chunked prefill, speculative verify) ------------------
def prefill_cost(w):
    """(algorithmic bytes, flops) of one pa_chunked_prefill launch: K+V of every
    context token of every (sequence, kv head) once, Q, out, tables, lengths;
    4 * D flops per (query row, visible key)."""
    q8 = getattr(w, "kv_dtype", "f16") in ("fp8", "int8")
    e = 1 if q8 else 2  # cache element bytes; queries and outputs are 16-bit
    lens = np.asarray(w.context_lens, dtype=np.int64)
    ql = np.asarray(w.q_lens, dtype=np.int64)
    kv = int(lens.sum()) * w.Hkv * w.D * 2 * e + (int(lens.sum()) * 8 if q8 else 0)
    io = w.T * w.Hq * w.D * 2 * 2
    meta = int(((lens + 15) // 16).sum()) * 4 + len(lens) * 8 + 4
    # visible keys of query i of sequence b: L_b - n_b + i + 1
    keys = int(sum(n * (L - n) + n * (n + 1) // 2 for L, n in zip(lens, ql)))
    return kv + io + meta, 4 * w.D * w.Hq * keys


class PrefillStep:
    """One step: pa_cache_write of every query token's K/V into the slots the
    block manager assigned, then pa_chunked_prefill over the paged context.
    The block manager admits each sequence's prior context and appends its
    chunk once at set-up; every step rewrites the same slots with the same
    values, so each timed step sees the same workload."""

    def __init__(self, w, split_tokens, device):
        import torch
        from paged_kv_cache_191_gb300 import ops
        self.torch, self.ops, self.L, self.w, self.dev = torch, ops, ops.lib(), w, device
        alloc = ops.BlockAllocator(w.num_blocks, w.free_order)
        slots = []
        for b in range(w.B):
            n, L = int(w.q_lens[b]), int(w.context_lens[b])
            alloc.alloc_seq(b, L - n)
            s, _ = alloc.append_tokens(b, n)
            slots.extend(s)
        self.cap = w.block_tables.shape[1]
        tables, lens = alloc.tables(list(range(w.B)), self.cap)
        if not np.array_equal(tables, w.block_tables) or not np.array_equal(lens, w.context_lens):
            raise RuntimeError("block manager tables differ from the workload's")
        slots = np.asarray(slots, dtype=np.int64)
        blk, row = slots // 16, slots % 16
        # the rows the chunk writes are the values the pool holds there
        new_k = w.k_pool[blk, :, row, :].contiguous()
        new_v = w.v_pool[blk, :, row, :].contiguous()
        self.q8 = w.kv_dtype in ("fp8", "int8")
        self.ks = self.vs = None
        if self.q8:  # the whole pool quantised on the device (set-up, not timed)
            N, H, _, D = w.k_pool.shape
            cdt = torch.int8 if w.kv_dtype == "int8" else torch.uint8
            self.kc = torch.zeros((N, H, 16, D), dtype=cdt, device=device)
            self.vc = torch.zeros_like(self.kc)
            self.ks = torch.zeros((N, 16), dtype=torch.float32, device=device)
            self.vs = torch.zeros_like(self.ks)
            ops.cache_write(w.k_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(device),
                            w.v_pool.permute(0, 2, 1, 3).reshape(N * 16, H, D).contiguous().to(device),
                            torch.arange(N * 16, dtype=torch.int64, device=device), self.kc, self.vc, self.ks,
                            self.vs)
        else:
            self.kc, self.vc = w.k_pool.to(device), w.v_pool.to(device)
        self.q = w.q.to(device)
        self.new_k, self.new_v = new_k.to(device), new_v.to(device)
        self.h_q, self.h_k, self.h_v = w.q.pin_memory(), new_k.pin_memory(), new_v.pin_memory()
        self.slots = torch.from_numpy(slots).to(device)
        self.q_start = torch.from_numpy(w.q_start.astype(np.int32)).to(device)
        self.tables = torch.from_numpy(tables.astype(np.int32)).to(device)
        self.lens = torch.from_numpy(lens.astype(np.int32)).to(device)
        self.out = torch.empty_like(self.q)
        self.max_len = int(lens.max())
        self.max_q = int(w.q_lens.max())
        self.split = split_tokens
        desc = ops.cache_desc(self.kc)
        self.ws_bytes = int(self.L.pa_chunked_prefill_workspace_size(w.T, w.B, w.Hq, self.max_q, self.max_len,
                                                                     C.byref(desc), split_tokens))
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        self.bytes, self.flops = prefill_cost(w)
        self.write_bytes = 2 * w.T * w.Hkv * w.D * (2 + (1 if self.q8 else 2)) + w.T * (16 if self.q8 else 8)

    def enqueue(self, stream, ev=None, q=None, k=None, v=None):
        ops = self.ops
        ops.cache_write(k if k is not None else self.new_k, v if v is not None else self.new_v, self.slots,
                        self.kc, self.vc, self.ks, self.vs, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        ops.chunked_prefill(q if q is not None else self.q, self.q_start, self.kc, self.vc, self.tables,
                            self.lens, self.max_len, self.max_q, self.w.scale, out=self.out, workspace=self.ws,
                            split_tokens=self.split, stream=stream, k_scale=self.ks, v_scale=self.vs)
        if ev is not None:
            ev[1].record(stream)

    def launches_per_step(self):
        """pa_cache_write, then what pa_chunked_prefill launches (its own count)."""
        w = self.w
        return 1 + self.ops.chunked_prefill_plan_info(w.T, w.B, w.Hq, self.max_q, self.max_len, self.kc, self.split)[3]


def _prefill_oracle_task(task):
    from oracle.attention import paged_prefill
    q, qs, kb, vb, L, scale, kvs = task[:7]
    rows = task[7] if len(task) > 7 else None  # a subset of (token, head) rows
    tab = np.arange(kb.shape[0], dtype=np.int64)[None, :]
    paged_prefill(q, qs, kb, vb, tab, np.array([L]), scale,
                  k_scale=kvs[0] if kvs else None, v_scale=kvs[1] if kvs else None, rows=rows)
    return L


def _quantise_prefill_task(task):
    """A task's f16 context blocks as 1-byte codes + per-token scales, by the
    oracle's quantiser (the cache write of an FP8 / INT8 cache)."""
    from oracle.cache_ops import quantize_rows
    q, qs, kb, vb, L, scale, fmt = task
    N, H, _, D = kb.shape
    cdt = np.int8 if fmt == "int8" else np.uint8
    out = []
    for blk in (kb, vb):
        c, s = quantize_rows(blk.transpose(0, 2, 1, 3).reshape(N * 16, H, D), cdt)
        out.append((c.reshape(N, 16, H, D).transpose(0, 2, 1, 3).copy(), s.reshape(N, 16)))
    return (q, qs, out[0][0], out[1][0], L, scale, (out[0][1], out[1][1]))


def prefill_oracle_tasks(w, codes=None):
    """Per-sequence oracle inputs (that sequence's blocks and query tokens);
    codes = (k codes, v codes, k scales, v scales) for a 1-byte cache."""
    from paged_kv_cache_191_gb300.workloads import BLOCK
    tasks, per = [], []
    qs = w.q_start
    for b in range(w.B):
        L, n = int(w.context_lens[b]), int(w.q_lens[b])
        blocks = w.block_tables[b][: -(-L // BLOCK)]
        f = (lambda t: t.float().numpy() if str(t.dtype) == "torch.bfloat16" else t.numpy())
        if codes is not None:
            kb, vb, kvs = codes[0][blocks], codes[1][blocks], (codes[2][blocks], codes[3][blocks])
        else:
            kb, vb, kvs = f(w.k_pool[blocks]), f(w.v_pool[blocks]), None
        tasks.append((f(w.q[qs[b]:qs[b + 1]]), [0, n], kb, vb, L, w.scale, kvs))
        sub = type("S", (), {})()
        sub.context_lens, sub.q_lens, sub.Hkv, sub.Hq, sub.D, sub.T = [L], [n], w.Hkv, w.Hq, w.D, n
        sub.kv_dtype = w.kv_dtype
        per.append(prefill_cost(sub)[0])
    return tasks, per


def run_prefill(args, rank, world, local_rank):
    import torch
    from paged_kv_cache_191_gb300 import workloads as W
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.PREFILL_CONFIGS[args.config]()
    st = PrefillStep(w, args.split, dev)
    stream = torch.cuda.Stream(device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st.enqueue(stream)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        gc_was = gc.isenabled()
        gc.disable()  # no collector pause between a launch's start event and its submission
        wall0 = time.time()
        t0e.record(stream)
        for i in range(args.steps):
            st.enqueue(stream, evs[i])
        t1e.record(stream)
        stream.synchronize()
        wall1 = time.time()
        if gc_was:
            gc.enable()
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    errs = st.ops.device_errors(clear=True)
    if errs:
        raise RuntimeError(f"device error flags {errs:#x} during the benchmark")
    local_s = t0e.elapsed_time(t1e) / 1e3
    k_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    step_bytes = st.bytes + st.write_bytes
    max_s, tot_bytes = aggregate(local_s, float(step_bytes * args.steps), world)
    _, tot_tokens = aggregate(local_s, float(w.T * args.steps), world)

    # e2e: public API with pinned host q / new K/V in and the output back, synced per step
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    hout = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(st.q), torch.empty_like(st.new_k), torch.empty_like(st.new_v)
    with torch.cuda.stream(stream):
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            dq.copy_(st.h_q, non_blocking=True)
            dk.copy_(st.h_k, non_blocking=True)
            dv.copy_(st.h_v, non_blocking=True)
            st.enqueue(stream, q=dq, k=dk, v=dv)
            hout.copy_(st.out, non_blocking=True)
            stream.synchronize()
        t1 = time.perf_counter()
    h2d = sum(t.numel() * t.element_size() for t in (st.h_q, st.h_k, st.h_v))
    e2e = {"value": round(step_bytes * n_e2e / (t1 - t0) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * hout.element_size()),
           "steps": n_e2e, "tokens_per_s": round(w.T * n_e2e / (t1 - t0), 1),
           "api": "paged_kv_cache_191_gb300.ops (pinned host buffers, stream sync per step)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tasks, per = prefill_oracle_tasks(w, (st.kc.cpu().numpy(), st.vc.cpu().numpy(), st.ks.cpu().numpy(),
                                              st.vs.cpu().numpy()) if st.q8 else None)
        cores = cpu_cores()
        order = sorted(range(w.B), key=lambda b: -int(w.q_lens[b]) * int(w.context_lens[b]))
        with _pool(cores) as pool:
            t0 = time.perf_counter()
            done_b = done_t = 0
            k = 0
            while time.perf_counter() - t0 < args.cpu_seconds and k < w.B:
                idx = order[k:k + cores]
                pool.map(_prefill_oracle_task, [tasks[i] for i in idx], chunksize=1)
                done_b += sum(per[i] for i in idx)
                done_t += sum(int(w.q_lens[i]) for i in idx)
                k += len(idx)
            t1 = time.perf_counter()
        cpu = {"value": round(done_b / (t1 - t0) / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{k} of {w.B} sequences of {w.name} (all heads, heaviest first), float64 NumPy "
                         f"oracle, spawn pool of {cores} single-threaded workers",
               "tokens_per_s": round(done_t / (t1 - t0), 2)}
    peak, peak_kind = hbm_peak()
    achieved = st.bytes / (k_ms / 1e3) / 1e9
    tflops = st.flops / (k_ms / 1e3) / 1e12
    res = {
        "metric": METRIC_PREFILL,
        "value": round(tot_bytes / max_s / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.kv_dtype + "+f32acc",
        "data": "synthetic",
        "config": {
            "workload": w.name, "sequences": w.B, "query_tokens": w.T, "q_heads": w.Hq, "kv_heads": w.Hkv,
            "head_dim": w.D, "block_size": 16, "kv_dtype": w.kv_dtype,
            "q_lens": f"{int(w.q_lens.min())}..{int(w.q_lens.max())}",
            "context_lens": f"{int(w.context_lens.min())}..{int(w.context_lens.max())} "
                            f"(mean {w.context_lens.mean():.0f}), chunk K/V rewritten every step",
            "split_tokens": args.split or "auto",
            "l2": f"no flush: K+V per step {st.bytes / 1e6:.0f} MB vs 129 MB L2",
            "parallelism": f"replicas x{world}",
        },
        "tokens_per_s": round(tot_tokens / max_s, 1),
        "tflops_attention": round(tflops, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind, "traffic": None,
                     "intensity_flop_per_byte": round(st.flops / st.bytes, 1),
                     "kernel": "pa_chunked_prefill (prefill_main + prefill_reduce)",
                     "bytes_per_launch": int(st.bytes), "flops_per_launch": int(st.flops),
                     "launch_ms": round(k_ms, 5)},
        "e2e": e2e,
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clocks.summary([(wall0, wall1)]),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(res), flush=True)


# ---- continuous-batching serving loop -------------------------------------------------
def run_serving(args, rank, world, local_rank):
    """K iterations of the serving loop after W warm-up iterations: the C++
    scheduler's step on the host, one H2D copy of its decisions, swap-out,
    cache write, multi-token attention, swap-in on the device.  Requests keep
    arriving (Poisson) for the whole run."""
    import torch
    from paged_kv_cache_191_gb300 import workloads as W
    from paged_kv_cache_191_gb300.serving import ServingLoop
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    tr = W.serving_llama7b()
    tdt = W.KV_TORCH[tr.kv_dtype]
    loop = ServingLoop(tr.num_blocks, tr.host_blocks, tr.Hkv, tr.Hq, tr.D, tdt, tr.max_batch, tr.max_tokens,
                       tr.max_context, device=dev, split_tokens=args.split)
    T_max = tr.max_batch + tr.max_tokens
    rng = W.rng_for(tr.seed)
    q = W.randn(rng, (T_max, tr.Hq, tr.D), tdt).to(dev)
    kn = W.randn(rng, (T_max, tr.Hkv, tr.D), tdt).to(dev)
    vn = W.randn(rng, (T_max, tr.Hkv, tr.D), tdt).to(dev)
    stream = torch.cuda.Stream(device=dev)
    att = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stats = {"tokens": 0, "prefill_tokens": 0, "decode_tokens": 0, "swap_out_blocks": 0, "swap_in_blocks": 0,
             "recomputed": 0, "finished": 0, "kv_bytes": 0, "flops": 0, "attn_launches": 0}
    e = 2
    clocks = ClockSampler(local_rank)
    clocks.start()
    it = 0

    def one(timed_i=None):
        nonlocal it
        for rid, p, m in tr.arrivals(it):
            loop.add(rid, p, m)
        st = loop.step(q, kn, vn, stream=stream, attn_events=att[timed_i] if timed_i is not None else None,
                       decisions=False)
        it += 1
        return st

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.time()
        host0 = time.perf_counter()
        t0e.record(stream)
        timed_attn = []
        sc = loop.sched
        v_kinds = np.ctypeslib.as_array(sc._kinds)
        v_starts = np.ctypeslib.as_array(sc._starts)
        v_lens = np.ctypeslib.as_array(sc._lens)
        o = sc._o
        for i in range(args.steps):
            st = one(i)
            n_it = st["n_items"]
            kinds, s0, n = v_kinds[:n_it], v_starts[:n_it].astype(np.int64), v_lens[:n_it].astype(np.int64)
            n_dec = int((kinds == 1).sum())
            stats["tokens"] += st["T"]
            stats["decode_tokens"] += n_dec
            stats["swap_out_blocks"] += o.n_swap_out
            stats["swap_in_blocks"] += o.n_swap_in
            stats["recomputed"] += o.n_recomputed
            stats["finished"] += o.n_finished
            timed_attn.append(i)
            if st["T"]:
                stats["kv_bytes"] += int((s0 + n).sum()) * tr.Hkv * tr.D * 2 * e + st["T"] * tr.Hq * tr.D * 2 * e
                stats["flops"] += int(4 * tr.D * tr.Hq * (n * s0 + n * (n + 1) // 2).sum())
                # decode_main (+ decode_reduce), cache write + prefill_main (+ prefill_reduce), swaps
                stats["attn_launches"] += (2 if n_dec else 0) + (3 if n_dec < n_it else 0) + \
                    (1 if o.n_swap_out else 0) + (1 if o.n_swap_in else 0)
        t1e.record(stream)
        host1 = time.perf_counter()
        stream.synchronize()
        wall1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    clocks.stop()
    stats["prefill_tokens"] = stats["tokens"] - stats["decode_tokens"]
    from paged_kv_cache_191_gb300 import ops
    errs = ops.device_errors(clear=True)
    if errs:
        raise RuntimeError(f"device error flags {errs:#x} during the benchmark")
    local_s = t0e.elapsed_time(t1e) / 1e3

    # e2e: the same loop with this iteration's queries and new K/V rows copied
    # from pinned host memory and the attention output read back, synced
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    hq, hk, hv = q.cpu().pin_memory(), kn.cpu().pin_memory(), vn.cpu().pin_memory()
    hout = torch.empty((T_max, tr.Hq, tr.D), dtype=tdt).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(kn), torch.empty_like(vn)
    e2e_tokens = h2d = d2h = 0
    with torch.cuda.stream(stream):
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            for rid, p, m in tr.arrivals(it):
                loop.add(rid, p, m)
            # plan first: the iteration's T new tokens are known before their
            # rows are copied, as a model producing them would need
            T = loop.plan()
            dq[:T].copy_(hq[:T], non_blocking=True)
            dk[:T].copy_(hk[:T], non_blocking=True)
            dv[:T].copy_(hv[:T], non_blocking=True)
            loop.launch(dq, dk, dv, stream=stream)
            it += 1
            if T:
                hout[:T].copy_(loop.out[:T], non_blocking=True)
            stream.synchronize()
            e2e_tokens += T
            h2d += T * (tr.Hq + 2 * tr.Hkv) * tr.D * e + loop.meta_bytes
            d2h += T * tr.Hq * tr.D * e
        t1 = time.perf_counter()

    attn_s = sum(att[i][0].elapsed_time(att[i][1]) for i in timed_attn) / 1e3
    max_s, tot_tokens = aggregate(local_s, float(stats["tokens"]), world)
    peak, peak_kind = hbm_peak()
    achieved = stats["kv_bytes"] / attn_s / 1e9 if attn_s else 0.0
    res = {
        "metric": METRIC_SERVING,
        "value": round(tot_tokens / max_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": tr.kv_dtype + "+f32acc",
        "data": "synthetic",
        "config": {"workload": tr.name, "q_heads": tr.Hq, "kv_heads": tr.Hkv, "head_dim": tr.D,
                   "gpu_blocks": tr.num_blocks, "host_blocks": tr.host_blocks, "max_batch": tr.max_batch,
                   "max_tokens_per_iteration": tr.max_tokens, "arrivals_per_iteration": tr.rate,
                   "prompt": f"log-uniform {tr.prompt_min}..{tr.prompt_max}",
                   "output": f"uniform {tr.out_min}..{tr.out_max}", "split_tokens": args.split or "auto",
                   "parallelism": f"replicas x{world}"},
        "iteration_stats": stats,
        "host_us_per_step": round((host1 - host0) * 1e6 / args.steps, 2),
        "device_ms_per_step": round(attn_s * 1e3 / args.steps, 5),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind, "traffic": None,
                     "kernel": "device work of pa_serve_step: staging copy, swaps, decode_main(+reduce) with the "
                               "fused write for decode items, cache write + prefill_main(+reduce) for chunks",
                     "tflops": round(stats["flops"] / attn_s / 1e12, 2) if attn_s else 0.0},
        "e2e": {"value": round(e2e_tokens / (t1 - t0), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d / n_e2e),
                "d2h_bytes_per_step": int(d2h / n_e2e), "steps": n_e2e,
                "api": "paged_kv_cache_191_gb300.serving.ServingLoop plan / launch: the iteration's q / K / V "
                       "rows in from pinned host memory, its attention output back, stream sync per iteration"},
        "gpu_launches": int(stats["attn_launches"]),
        "clocks": clocks.summary([(wall0, wall1)]),
        "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(res), flush=True)


# ---- CPU oracle (baseline and reference arm) --------------------------------------
def _oracle_task(task):
    import numpy as np  # noqa: F811
    from oracle.attention import paged_decode
    q, kb, vb, n, scale, ks, vs = task
    tab = np.arange(kb.shape[0], dtype=np.int64)[None, :]
    paged_decode(q[None], kb, vb, tab, np.array([n]), scale, ks, vs)
    return n


def oracle_tasks(w, seqs, codes=None):
    """Per-sequence oracle inputs: that sequence's blocks (de-duplicated pool view)."""
    from paged_kv_cache_191_gb300.workloads import BLOCK
    tasks = []
    for b in seqs:
        n = int(w.context_lens[b])
        blocks = w.block_tables[b][: -(-n // BLOCK)]
        kb = w.k_pool[blocks]
        vb = w.v_pool[blocks]
        kb = kb.float().numpy() if str(kb.dtype) == "torch.bfloat16" else kb.numpy()
        vb = vb.float().numpy() if str(vb.dtype) == "torch.bfloat16" else vb.numpy()
        q = w.q[b].float().numpy() if str(w.q.dtype) == "torch.bfloat16" else w.q[b].numpy()
        if codes is not None:  # "fp8" or "int8": the oracle's own quantiser of that format
            from oracle.cache_ops import quantize_rows
            H, D = kb.shape[1], kb.shape[3]
            cdt = np.int8 if codes == "int8" else np.uint8
            kcodes, ks = quantize_rows(kb.transpose(0, 2, 1, 3).reshape(-1, H, D), cdt)
            vcodes, vs = quantize_rows(vb.transpose(0, 2, 1, 3).reshape(-1, H, D), cdt)
            kb = kcodes.reshape(-1, 16, H, D).transpose(0, 2, 1, 3).copy()
            vb = vcodes.reshape(-1, 16, H, D).transpose(0, 2, 1, 3).copy()
            tasks.append((q, kb, vb, n, w.scale, ks.reshape(-1, 16), vs.reshape(-1, 16)))
        else:
            tasks.append((q, kb, vb, n, w.scale, None, None))
    return tasks


def _pool(cores):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    for k in env_keys:
        os.environ[k] = "1"
    return ctx.Pool(cores)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds):
    """The oracle as it stands over whole sequences of the workload, in a spawn
    pool over the host cores, repeated until about `seconds` have passed."""
    cores = cpu_cores()
    seqs = list(range(w.B))
    q8 = w.kv_dtype in ("fp8", "int8")
    tasks = oracle_tasks(w, seqs, codes=w.kv_dtype if q8 else None)
    e = 1 if q8 else 2
    per_seq = [decode_bytes([int(w.context_lens[b])], w.Hq, w.Hkv, w.D, e, 2, 2) for b in seqs]
    with _pool(cores) as pool:
        t0 = time.perf_counter()
        done_b = 0
        rounds = 0
        while True:
            pool.map(_oracle_task, tasks, chunksize=1)
            done_b += sum(per_seq)
            rounds += 1
            if time.perf_counter() - t0 >= seconds or rounds >= 50:
                break
        t1 = time.perf_counter()
    return {"value": round(done_b / (t1 - t0) / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{rounds} pass(es) over all {w.B} sequences x {w.Hq} heads of {w.name} "
                      f"(float64 NumPy oracle, spawn pool of {cores} single-threaded workers)",
            "tokens_per_s": round(rounds * w.B / (t1 - t0), 2)}


def _per_kv_head(tasks, per):
    """Decode oracle tasks split per kv head: (G query heads, one kv head's
    blocks), each carrying its share of the sequence's algorithmic bytes."""
    out, out_per = [], []
    for (q, kb, vb, n, scale, ks, vs), p in zip(tasks, per):
        Hkv = kb.shape[1]
        G = q.shape[0] // Hkv
        for g in range(Hkv):
            out.append((q[g * G:(g + 1) * G], kb[:, g:g + 1], vb[:, g:g + 1], n, scale, ks, vs))
            out_per.append(p / Hkv)
    return out, out_per


def _per_head_slice(tasks, per, G, slice_tokens=64):
    """Multi-token oracle tasks split per (kv head, slice of query tokens):
    the rows of that slice for that kv head's G query heads."""
    out, out_per = [], []
    for (q, qs, kb, vb, L, scale, kvs), p in zip(tasks, per):
        n, Hkv = q.shape[0], kb.shape[1]
        for g in range(Hkv):
            qg, kbg, vbg = q[:, g * G:(g + 1) * G], kb[:, g:g + 1], vb[:, g:g + 1]
            for t0 in range(0, n, slice_tokens):
                t1 = min(n, t0 + slice_tokens)
                rows = [(t, h) for t in range(t0, t1) for h in range(G)]
                out.append((qg, qs, kbg, vbg, L, scale, kvs, rows))
                out_per.append(p / Hkv * (t1 - t0) / n)
    return out, out_per


def _bounded_oracle_loop(pool, fn, tasks, per, steps, warmup, cores, total_s=150.0):
    """W + K steps of the oracle over the tasks (cycled), each step as many
    tasks as one calibrated round of the pool fits in total_s / (W + K)
    seconds, so the whole run stays near total_s whatever K is (at one task
    per step at least).  Returns (bytes done, seconds, tasks per step)."""
    budget = total_s / max(1, steps + warmup)
    pool.map(fn, tasks[:cores], chunksize=1)  # workers start and import the oracle
    t = time.perf_counter()
    pool.map(fn, [tasks[(cores + j) % len(tasks)] for j in range(cores)], chunksize=1)
    round_s = time.perf_counter() - t  # one task on each worker
    n = int(max(1, min(len(tasks), cores * budget / max(round_s, 1e-6))))
    k = 0
    for _ in range(warmup):
        pool.map(fn, [tasks[(k + j) % len(tasks)] for j in range(n)], chunksize=1)
        k += n
    done_b = 0.0
    t0 = time.perf_counter()
    for _ in range(steps):
        idx = [(k + j) % len(tasks) for j in range(n)]
        pool.map(fn, [tasks[i] for i in idx], chunksize=1)
        done_b += sum(per[i] for i in idx)
        k += n
    return done_b, time.perf_counter() - t0, n


def run_reference_prefill(args, world):
    """Reference arm for the multi-token workloads: the oracle over a bounded
    sample of sequences per step, on host cores."""
    from paged_kv_cache_191_gb300 import workloads as W
    w = W.PREFILL_CONFIGS[args.config]()
    tasks, per = prefill_oracle_tasks(w)
    cores = cpu_cores()
    with _pool(cores) as pool:
        if w.kv_dtype in ("fp8", "int8"):  # the cache's codes and scales (set-up, not timed)
            tasks = pool.map(_quantise_prefill_task, [t[:6] + (w.kv_dtype,) for t in tasks], chunksize=1)
        keep = [i for i, t in enumerate(tasks) if t[0].shape[0] > 0]
        tasks, per = _per_head_slice([tasks[i] for i in keep], [per[i] for i in keep], w.Hq // w.Hkv)
        done_b, secs, n_per_step = _bounded_oracle_loop(pool, _prefill_oracle_task, tasks, per, args.steps,
                                                        args.warmup, cores)
    t0, t1 = 0.0, secs
    val = round(done_b / (t1 - t0) / 1e9, 4)
    sample = (f"each step: {n_per_step} of the {len(tasks)} (sequence, kv head, 64-token slice) tasks of "
              f"{w.name}, cycled; float64 NumPy oracle, spawn pool of {cores} workers")
    print(json.dumps({
        "impl": "reference", "metric": METRIC_PREFILL, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((t1 - t0) * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sequences": w.B, "query_tokens": w.T, "q_heads": w.Hq,
                   "kv_heads": w.Hkv, "head_dim": w.D, "kv_dtype": w.kv_dtype, "parallelism": "host cores"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def shared_prefix_view(w):
    """The shared-prefix workload's first step as a plain decode batch, built
    on the host block manager alone (every beam forked from its group's
    prompt, then grown by its tail)."""
    from types import SimpleNamespace
    from paged_kv_cache_191_gb300 import ops
    alloc = ops.BlockAllocator(w.num_blocks, w.free_order)
    roots = [10 ** 9 + g for g in range(w.groups)]
    for r in roots:
        alloc.alloc_seq(r, w.prompt_len)
    ids = list(range(w.B))
    alloc.fork_seqs([roots[i // w.beams] for i in ids], ids)
    tails = w.tail_lens.reshape(-1)
    for i in ids:
        alloc.append_tokens(i, int(tails[i]), want_slots=False)
    cap = -(-(w.prompt_len + int(tails.max())) // 16)
    tables, lens = alloc.tables(ids, cap)
    return SimpleNamespace(name=w.name, B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, kv_dtype="f16", context_lens=lens,
                           block_tables=tables, k_pool=w.k_pool, v_pool=w.v_pool, q=w.q, scale=w.scale)


def run_reference_serving(args, world):
    """Reference arm for the serving loop: the oracle scheduler over the same
    request trace, the oracle's cache writes and swaps on a host mirror of the
    pools, and the oracle's multi-token attention for each iteration's items
    (in order, until the step's time budget is spent), in one host process."""
    from oracle.attention import paged_prefill
    from oracle.scheduler import Scheduler as OSched
    from paged_kv_cache_191_gb300 import workloads as W
    tr = W.serving_llama7b()
    sched = OSched(tr.num_blocks, tr.max_batch, tr.max_tokens, tr.host_blocks)
    Hq, Hkv, D = tr.Hq, tr.Hkv, tr.D
    kc = np.zeros((tr.num_blocks, Hkv, 16, D), np.float16)
    vc = np.zeros_like(kc)
    kh = np.zeros((tr.host_blocks, Hkv, 16, D), np.float16)
    vh = np.zeros_like(kh)
    rng = np.random.default_rng(tr.seed)
    T_max = tr.max_batch + tr.max_tokens
    bq = rng.standard_normal((T_max, Hq, D)).astype(np.float16)
    bk = rng.standard_normal((T_max, Hkv, D)).astype(np.float16)
    bv = rng.standard_normal((T_max, Hkv, D)).astype(np.float16)
    budget = 150.0 / max(1, args.steps + args.warmup)
    scale = 1.0 / np.sqrt(D)
    it = 0

    def one():
        nonlocal it
        for rid, p, m in tr.arrivals(it):
            sched.add(rid, p, m)
        r = sched.step()
        it += 1
        for g, h in r.swap_out:
            kh[h], vh[h] = kc[g], vc[g]
        row = 0
        work = []
        for rid, kind, start, slots in r.items:
            sl = np.asarray(slots, dtype=np.int64)
            kc[sl // 16, :, sl % 16, :] = bk[row: row + len(sl)]
            vc[sl // 16, :, sl % 16, :] = bv[row: row + len(sl)]
            work.append((row, len(sl), start + len(sl), list(sched.alloc.tables[rid])))
            row += len(sl)
        t = time.perf_counter()
        done = 0.0
        G = Hq // Hkv
        for r0, n, L, tab in work:  # attention before the swap-ins, as on the device
            for g in range(Hkv):     # in (kv head, 64-token slice) pieces, within the step's budget
                for t0 in range(0, n, 64):
                    if time.perf_counter() - t > budget:
                        break
                    rows = [(x, h) for x in range(t0, min(n, t0 + 64)) for h in range(g * G, (g + 1) * G)]
                    paged_prefill(bq[r0: r0 + n], [0, n], kc, vc, np.asarray([tab]), np.array([L]), scale,
                                  rows=rows)
                    done += len(rows) / Hq  # in query tokens
        for h, g in r.swap_in:
            kc[g], vc[g] = kh[h], vh[h]
        return done

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    tokens = sum(one() for _ in range(args.steps))
    t1 = time.perf_counter()
    val = round(tokens / (t1 - t0), 2)
    sample = (f"{args.steps} iterations of {tr.name} after {args.warmup} warm-up: oracle scheduler, cache "
              f"writes and swaps in full, attention of each iteration's items in (kv head, 64-token slice) "
              f"pieces in order within {budget * 1e3:.1f} ms, one host process")
    print(json.dumps({
        "impl": "reference", "metric": METRIC_SERVING, "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round((t1 - t0) * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": tr.name, "q_heads": Hq, "kv_heads": Hkv, "head_dim": D, "parallelism": "host"},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args, rank, world):
    """Reference arm: the float64 CPU oracle on host cores, K bounded steps."""
    if rank != 0:
        return
    if args.config in PREFILL_CONFIGS:
        return run_reference_prefill(args, world)
    if args.config in SERVING_CONFIGS:
        return run_reference_serving(args, world)
    shared = args.config == "shared_prefix_16x4"
    sw = load_workload(args.config)
    w = shared_prefix_view(sw) if shared else sw
    cores = cpu_cores()
    fp8 = w.kv_dtype in ("fp8", "int8")
    e = 1 if fp8 else 2
    seqs = list(range(w.B))
    seqs = [b for b in seqs if int(w.context_lens[b]) > 0]
    tasks = oracle_tasks(w, seqs, codes=w.kv_dtype if fp8 else None)
    per = [decode_bytes([int(w.context_lens[b])], w.Hq, w.Hkv, w.D, e, 2, 2) for b in seqs]
    if shared:  # unique bytes: each beam carries a 1/beams share of its group's prompt
        tails = sw.tail_lens.reshape(-1)
        per = [decode_bytes([int(tails[b])], w.Hq, w.Hkv, w.D, e, 2, 2)
               + sw.prompt_len * w.Hkv * w.D * 2 * e / sw.beams for b in seqs]
    tasks, per = _per_kv_head(tasks, per)
    with _pool(cores) as pool:
        done_b, secs, n_per_step = _bounded_oracle_loop(pool, _oracle_task, tasks, per, args.steps, args.warmup,
                                                        cores)
    t0, t1 = 0.0, secs
    val = round(done_b / (t1 - t0) / 1e9, 4)
    sample = (f"each step: {n_per_step} of the {len(tasks)} (sequence, kv head) tasks of {w.name}, cycled; "
              f"float64 NumPy oracle, spawn pool of {cores} workers")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round((t1 - t0) * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
                   "head_dim": w.D, "kv_dtype": w.kv_dtype, "parallelism": "host cores"},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.config in PREFILL_CONFIGS:
            run_prefill(args, rank, world, local_rank)
        elif args.config in SERVING_CONFIGS:
            run_serving(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
