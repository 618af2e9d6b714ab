"""Tolerance used by the parity tests.

The layer's outputs are fp16.  The pass criterion (fp32 accumulation, fp16
I/O) is:
  * relative L2 error  ||gpu - ref|| / ||ref||            <= 5e-3, and
  * max_i |gpu_i - ref_i| / max(1, rms(ref row of i))     <= 2e-2,
where ref is the oracle's fp64 output before rounding.  The second is the
2e-2 absolute bound measured in units of the row's magnitude once that
magnitude exceeds 1: for outputs of size |y| >= 64 the fp16 rounding of the
output alone is up to 1/32, so an absolute 2e-2 bound would fail any
implementation there.  For rows with rms <= 1 it is the absolute bound.
"""
import numpy as np

REL_L2 = 5e-3
MAX_NORM = 2e-2


def stats(out16, ref64):
    got = np.asarray(out16).view(np.float16).astype(np.float64) \
        if np.asarray(out16).dtype == np.uint16 else np.asarray(out16, np.float64)
    ref = np.asarray(ref64, np.float64)
    d = got - ref
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    half_ulp = np.abs(ref).astype(np.float16).astype(np.float64)
    half_ulp = np.spacing(half_ulp.astype(np.float16)).astype(np.float64) / 2
    return dict(
        rel_l2=float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300)),
        max_norm=float(np.max(np.abs(d) / np.maximum(1.0, rms))),
        max_abs=float(np.max(np.abs(d))),
        max_over_half_ulp=float(np.max(np.abs(d) - half_ulp)),
    )


def assert_close(out16, ref64, what=""):
    s = stats(out16, ref64)
    assert s["rel_l2"] <= REL_L2 and s["max_norm"] <= MAX_NORM, "%s %s" % (what, s)
    return s
