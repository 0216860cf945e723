"""Shared checks for the GPU parity tests.

Tolerances are the ones the library promises per precision:
  ATTN_FP32  |gpu - ref| <= 1e-5 + 1e-4 |ref| elementwise; LSE slots within 1e-4.
  ATTN_TF32  max |gpu - ref| / max |V| <= 3e-3.
  ATTN_BF16  max |gpu - ref| / max |V| <= 2e-2.
"""
import numpy as np
import torch

FP32, TF32, BF16 = 0, 1, 2
NORM_TOL = {TF32: 3e-3, BF16: 2e-2}
# LSE tolerance of the tensor-core paths (not given by the target; derived from
# the operand rounding: relative operand error 2^-11 (TF32) / 2^-8 (bf16) times
# the largest score magnitude, floored at 1).
LSE_TOL = {TF32: 3e-3, BF16: 2e-2}


def dev(x):
    return x.to("cuda").contiguous()


def assert_out_close(got, ref, prec, vmax, where=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), where + ": non-finite output"
    err = np.abs(got - ref)
    if prec == FP32:
        bad = err > 1e-5 + 1e-4 * np.abs(ref)
        assert not bad.any(), "%s: %d elements out of tolerance, worst |err| %.3g at ref %.3g" % (
            where, int(bad.sum()), err.max(), ref.flat[int(np.argmax(err))])
    else:
        rel = err.max() / max(vmax, 1e-30)
        assert rel <= NORM_TOL[prec], "%s: max|err|/max|V| = %.3g > %.3g" % (where, rel, NORM_TOL[prec])


def assert_lse_close(got, ref, prec, smax=1.0, where=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    tol = 1e-4 if prec == FP32 else LSE_TOL[prec] * max(1.0, smax)
    assert err.max() <= tol, "%s: LSE max err %.3g > %.3g" % (where, err.max(), tol)


def tc_supported(H, G, D):
    """Shapes the tensor-core precisions accept: D in {64, 128} (layouts their
    kernels do not take run on the fp32 kernel)."""
    return D in (64, 128)
