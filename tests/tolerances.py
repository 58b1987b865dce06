"""Parity metric and tolerances shared by the tests.

max relative error of a tensor = max_i |got_i - ref_i| / max_i |ref_i|  (infinity-norm
relative error).  Bars: 1e-4 when the pool's state is fp32 and the compared tensor is
stored in fp32; 2e-2 when either is bf16 (a bf16 output carries its own rounding, and a
bf16-state pool runs bf16 tensor-core operands).
Integer, index and byte results are compared bit for bit instead.
"""
import numpy as np

TOL = {0: 1e-4, 1: 2e-2}  # keyed by dtype: 0 = fp32, 1 = bf16


def tol(state_dtype: int, tensor_dtype: int) -> float:
    return TOL[max(state_dtype, tensor_dtype)]


def max_rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    denom = float(np.max(np.abs(ref)))
    diff = float(np.max(np.abs(got - ref)))
    if denom == 0.0:
        return diff
    return diff / denom
