"""Oracle quantisation of one sequence's blocks, as a process-pool task.

Imports only NumPy and the oracle, so spawn workers start quickly and never
touch CUDA.  The blocks are written into a compact pool (block i of the
result is the i-th listed physical block) through the oracle's own cache
write, one token per slot.
"""
import numpy as np

from oracle.cache_ops import cache_write

BLOCK = 16


def quantise_blocks(task):
    """(k_blocks, v_blocks [n, H, 16, D] values, cache dtype) -> oracle
    (k codes, v codes [n, H, 16, D], k scales, v scales [n, 16])."""
    kb, vb, dtype = task
    n, H, _, D = kb.shape
    kin = np.ascontiguousarray(kb.transpose(0, 2, 1, 3)).reshape(n * BLOCK, H, D)
    vin = np.ascontiguousarray(vb.transpose(0, 2, 1, 3)).reshape(n * BLOCK, H, D)
    kc = np.zeros((n, H, BLOCK, D), dtype)
    ks = np.zeros((n, BLOCK), np.float32)
    return cache_write(kin, vin, np.arange(n * BLOCK), kc, kc.copy(), ks, ks.copy())
