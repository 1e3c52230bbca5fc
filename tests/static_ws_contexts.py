"""pa_decode_static_ws in more than one CUDA context, without torch.

Run as a child process by tests/test_zz_no_alloc.py (``python -m
tests.static_ws_contexts``).  Device memory comes from the driver API
(cuMemAlloc in whichever context is current), so the library is called in:

1. the device's primary context,
2. a second context created on the same device (its own copy of the
   library's device code, so the static array sits at another address), and
3. the primary context again after the second one is destroyed.

A static-scratch address cached from an earlier context would point into
memory that the current context does not own; the entry point must look the
address up again whenever the current context changes.  A cudaDeviceReset
gives the same situation (a new primary context); a second context makes it
without tearing down state the rest of the process holds.  The three outputs
must be bit-identical and match the float64 oracle within the f16
tolerance.  Prints "ok" and exits 0 on success.
"""
import ctypes as C
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle.attention import paged_decode  # noqa: E402

LIB = os.path.join(ROOT, "paged_kv_cache_191_gb300", "libpagedkv.so")
F16, F32 = 0, 3


class Desc(C.Structure):
    _fields_ = [("num_blocks", C.c_int32), ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("block_size", C.c_int32), ("kv_dtype", C.c_int32)]


def driver():
    cu = C.CDLL("libcuda.so.1")
    P, U64 = C.c_void_p, C.c_uint64
    cu.cuInit.argtypes = [C.c_uint]
    cu.cuDeviceGet.argtypes = [C.POINTER(C.c_int), C.c_int]
    cu.cuDevicePrimaryCtxRetain.argtypes = [C.POINTER(P), C.c_int]
    cu.cuDevicePrimaryCtxRelease_v2.argtypes = [C.c_int]
    cu.cuCtxSetCurrent.argtypes = [P]
    cu.cuCtxDestroy_v2.argtypes = [P]
    cu.cuCtxSynchronize.argtypes = []
    cu.cuMemAlloc_v2.argtypes = [C.POINTER(U64), C.c_size_t]
    cu.cuMemFree_v2.argtypes = [U64]
    cu.cuMemcpyHtoD_v2.argtypes = [U64, P, C.c_size_t]
    cu.cuMemcpyDtoH_v2.argtypes = [P, U64, C.c_size_t]
    return cu


def ok(rc, what):
    if rc != 0:
        raise SystemExit(f"{what} failed with CUresult {rc}")


def make_inputs():
    """B = 4 sequences, 8 q / 2 kv heads, head_dim 128, f16 N(0,1); lengths
    that split into several 256-token partitions, tables a seeded
    permutation of the pool."""
    rng = np.random.Generator(np.random.PCG64(2024))
    B, Hq, Hkv, D = 4, 8, 2, 128
    lens = np.array([700, 1500, 33, 2000], dtype=np.int32)
    nblk = (lens + 15) // 16
    num_blocks = int(nblk.sum()) + 5
    perm = rng.permutation(num_blocks)
    tables = np.full((B, int(nblk.max())), -1, dtype=np.int32)
    at = 0
    for b in range(B):
        tables[b, : nblk[b]] = perm[at: at + nblk[b]]
        at += nblk[b]
    q = rng.standard_normal((B, Hq, D), dtype=np.float32).astype(np.float16)
    kc = rng.standard_normal((num_blocks, Hkv, 16, D), dtype=np.float32).astype(np.float16)
    vc = rng.standard_normal((num_blocks, Hkv, 16, D), dtype=np.float32).astype(np.float16)
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, lens=lens, tables=tables, q=q, kc=kc, vc=vc,
                num_blocks=num_blocks, scale=1.0 / np.sqrt(D))


def run_in_current_context(cu, lib, x):
    """Allocate, upload, one pa_decode_static_ws call (legacy default stream),
    read back, free -- all in the context current on this thread."""
    out = np.empty((x["B"], x["Hq"], x["D"]), dtype=np.float32)
    host = {"q": x["q"], "kc": x["kc"], "vc": x["vc"], "bt": np.ascontiguousarray(x["tables"]),
            "cl": x["lens"], "out": out}
    dev = {}
    try:
        for k, a in host.items():
            p = C.c_uint64()
            ok(cu.cuMemAlloc_v2(C.byref(p), a.nbytes), "cuMemAlloc")
            dev[k] = p.value
            if k != "out":
                ok(cu.cuMemcpyHtoD_v2(dev[k], a.ctypes.data, a.nbytes), "cuMemcpyHtoD")
        desc = Desc(x["num_blocks"], x["Hkv"], x["D"], 16, F16)
        st = lib.pa_decode_static_ws(
            C.c_void_p(dev["q"]), F16, C.c_void_p(dev["kc"]), C.c_void_p(dev["vc"]), None, None,
            C.c_void_p(dev["bt"]), x["tables"].shape[1], C.c_void_p(dev["cl"]), int(x["lens"].max()),
            x["B"], x["Hq"], C.c_float(x["scale"]), C.c_void_p(dev["out"]), F32, C.byref(desc), 256, None)
        if st != 0:
            raise SystemExit(f"pa_decode_static_ws returned {st}: {lib.pa_last_error().decode()}")
        ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        flags = C.c_uint32()
        if lib.pa_device_errors(C.byref(flags), 1) != 0 or flags.value:
            raise SystemExit(f"device error word {flags.value:#x}")
        ok(cu.cuMemcpyDtoH_v2(out.ctypes.data, dev["out"], out.nbytes), "cuMemcpyDtoH")
    finally:
        for p in dev.values():
            cu.cuMemFree_v2(p)
    return out


def main():
    cu = driver()
    lib = C.CDLL(LIB)
    lib.pa_last_error.restype = C.c_char_p
    x = make_inputs()
    ok(cu.cuInit(0), "cuInit")
    dev = C.c_int()
    ok(cu.cuDeviceGet(C.byref(dev), 0), "cuDeviceGet")
    primary = C.c_void_p()
    ok(cu.cuDevicePrimaryCtxRetain(C.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ok(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    first = run_in_current_context(cu, lib, x)

    second_ctx = C.c_void_p()
    if hasattr(cu, "cuCtxCreate_v4"):
        cu.cuCtxCreate_v4.argtypes = [C.POINTER(C.c_void_p), C.c_void_p, C.c_uint, C.c_int]
        ok(cu.cuCtxCreate_v4(C.byref(second_ctx), None, 0, dev), "cuCtxCreate")
    else:
        cu.cuCtxCreate_v2.argtypes = [C.POINTER(C.c_void_p), C.c_uint, C.c_int]
        ok(cu.cuCtxCreate_v2(C.byref(second_ctx), 0, dev), "cuCtxCreate")
    ok(cu.cuCtxSetCurrent(second_ctx), "cuCtxSetCurrent")
    second = run_in_current_context(cu, lib, x)
    ok(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    ok(cu.cuCtxDestroy_v2(second_ctx), "cuCtxDestroy")
    third = run_in_current_context(cu, lib, x)
    cu.cuDevicePrimaryCtxRelease_v2(dev)

    if not (np.array_equal(first, second) and np.array_equal(first, third)):
        raise SystemExit("outputs differ between contexts")
    ref = paged_decode(x["q"], x["kc"], x["vc"], x["tables"], x["lens"], x["scale"])
    err = float(np.abs(first - ref).max())
    if not err <= 2e-3:
        raise SystemExit(f"max abs error {err:.3e} against the oracle")
    print("ok", err)


if __name__ == "__main__":
    main()
