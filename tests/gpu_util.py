"""Helpers shared by the GPU parity tests (device moves, oracle inputs)."""
import numpy as np
import pytest
import torch

TOL = {"f16": 2e-3, "bf16": 2e-3, "fp8": 2e-2, "int8": 2e-2}

requires_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def np_exact(t):
    """CPU numpy copy of a tensor with every value exact (bf16 -> float32)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def half_ulp(x, dtype):
    """Half a unit in the last place of |x| in a 16-bit float dtype."""
    mant = 10 if dtype == torch.float16 else 7
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - mant)


def assert_close(got, want, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert worst <= tol, f"{what}: max abs err {worst:.3e} > {tol:.1e}"
    return worst
