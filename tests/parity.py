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

A third figure measures the error in fp16 rounding units: the part of
|gpu - ref| beyond the half ulp of fp16 that rounding the output to fp16
costs any implementation, over max(1, rms(row)), must stay within
BEYOND_ROUNDING = 5e-3 (the relative-L2 bound, applied per element).  It is
what remains of the error once the output's own rounding is taken out: the
fp32 accumulation, the fp16 SwiGLU activations between the projections and
the fp16 weights of the large-batch GEMM.
"""
import json
import os

import numpy as np

REL_L2 = 5e-3
MAX_NORM = 2e-2
BEYOND_ROUNDING = 5e-3


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
        beyond_rounding=float(np.max(np.maximum(np.abs(d) - half_ulp, 0.0)
                                     / np.maximum(1.0, rms))),
    )


def assert_close(out16, ref64, what=""):
    s = stats(out16, ref64)
    log = os.environ.get("QE_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(dict(s, what=what)) + "\n")
    assert s["rel_l2"] <= REL_L2 and s["max_norm"] <= MAX_NORM, "%s %s" % (what, s)
    assert s["beyond_rounding"] <= BEYOND_ROUNDING, "%s %s" % (what, s)
    return s
