"""pa_decode_static_ws: decode for callers that cannot allocate device memory.

Some callers of this library cannot allocate device memory when they decode
(a plugin inside an engine whose allocator owns the device and offers no
scratch hook, or a latency-critical loop where cudaMalloc/cudaFree would
stall).  pa_decode_static_ws keeps the split-K partials in a static device
array of the library instead of a caller workspace.  These tests call it
through the C ABI and check it against pa_decode with a caller-provided
workspace, on two calls in a row (the array keeps the previous call's
contents), plus the rejection of shapes that do not fit the array.

The file is named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle.attention import paged_decode
from paged_kv_cache_191_gb300 import ops, workloads as W
from tests.gpu_util import TOL, np_exact, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]
DEV = "cuda"


def _inputs(w):
    return (w.q.to(DEV), w.k_pool.to(DEV), w.v_pool.to(DEV),
            torch.from_numpy(w.block_tables).to(DEV), torch.from_numpy(w.context_lens).to(DEV))


def _decode_c(name, w, dev_in, out, split, ws=None):
    q, kc, vc, bt, cl = dev_in
    desc = ops.cache_desc(kc)
    args = [q.data_ptr(), ops._TORCH_DT[q.dtype], kc.data_ptr(), vc.data_ptr(), None, None,
            bt.data_ptr(), bt.shape[1], cl.data_ptr(), int(w.context_lens.max()), w.B, w.Hq,
            C.c_float(w.scale), out.data_ptr(), ops.F32, C.byref(desc)]
    if name == "pa_decode":
        args += [ws.data_ptr() if ws is not None else None, ws.numel() if ws is not None else 0]
    args += [split, C.c_void_p(torch.cuda.current_stream().cuda_stream)]
    return getattr(ops.lib(), name)(*args)


def test_static_scratch_matches_caller_workspace_on_two_calls():
    for call, (seed, dt, split) in enumerate([(61, "f16", 256), (62, "bf16", 128)]):
        w = W.random_small(seed, B=6, Hq=16, Hkv=2, D=128, kv_dtype=dt, max_len=2500, min_len=600)
        dev_in = _inputs(w)
        need = ops.decode_workspace_size(w.B, w.Hq, int(w.context_lens.max()), dev_in[1], split)
        assert 0 < need <= 32 * 1024 * 1024  # several partitions: the scratch is used
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        ref_out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=DEV)
        st_out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
        assert _decode_c("pa_decode", w, dev_in, ref_out, split, ws) == ops.PA_OK
        assert _decode_c("pa_decode_static_ws", w, dev_in, st_out, split) == ops.PA_OK, \
            ops.lib().pa_last_error()
        torch.cuda.synchronize()
        a, b = ref_out.cpu().numpy(), st_out.cpu().numpy()
        assert np.all(np.isfinite(b)), f"call {call}: output not fully written"
        assert np.abs(a - b).max() <= TOL[dt], f"call {call}: differs from pa_decode"
        ref = paged_decode(np_exact(w.q), np_exact(w.k_pool), np_exact(w.v_pool), w.block_tables,
                           w.context_lens, w.scale)
        assert np.abs(b - ref).max() <= TOL[dt], f"call {call}: differs from the oracle"


def test_shapes_beyond_the_static_array_are_rejected():
    w = W.random_small(63, B=2, Hq=8, Hkv=8, D=128, kv_dtype="f16", max_len=40, min_len=20)
    dev_in = _inputs(w)
    q, kc, vc, bt, cl = dev_in
    desc = ops.cache_desc(kc)
    out = torch.zeros((w.B, w.Hq, w.D), dtype=torch.float32, device=DEV)
    big_b, big_ctx = 256, 1 << 20   # 1024 partitions of 1024 tokens: ~1 GB of partials
    assert ops.decode_workspace_size(big_b, w.Hq, big_ctx, kc, 1024) > 32 * 1024 * 1024
    st = ops.lib().pa_decode_static_ws(q.data_ptr(), ops.F16, kc.data_ptr(), vc.data_ptr(), None, None,
                                       bt.data_ptr(), bt.shape[1], cl.data_ptr(), big_ctx, big_b, w.Hq,
                                       C.c_float(w.scale), out.data_ptr(), ops.F32, C.byref(desc), 1024,
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ops.PA_ERR_INVALID
    assert b"static array" in ops.lib().pa_last_error()
    torch.cuda.synchronize()
    assert not out.any(), "a rejected call must launch nothing"


def test_static_scratch_follows_the_current_context():
    """The array's address is per context: calls in the primary context, in a
    second context on the same device, and in the primary context again must
    each use their own context's copy (a child process drives the contexts
    through the driver API, without torch)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "tests.static_ws_contexts"], cwd=root, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
