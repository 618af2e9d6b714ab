"""Independent test-side arithmetic used to pin the oracle.

Nothing here calls the oracle or the CUDA path.  Each helper restates a
definition with a different mechanism than the oracle uses (numpy bit
operations instead of C loops, Python rationals instead of 128-bit integers,
numpy matrix products instead of per-row loops), so an error in either shows
up as a mismatch.
"""
from fractions import Fraction

import numpy as np


def unpack(codes: np.ndarray, K: int, wbits: int) -> np.ndarray:
    """Canonical packed codes [..., K*wbits/8] -> integer codes [..., K]."""
    codes = np.asarray(codes, np.uint8)
    per = 8 // wbits
    mask = (1 << wbits) - 1
    fields = [(codes >> (wbits * i)) & mask for i in range(per)]
    out = np.stack(fields, axis=-1)  # [..., K/per, per]: element k = byte k//per, field k%per
    return out.reshape(codes.shape[:-1] + (K,))


def dequant(codes, scales, zeros, K, wbits, group=128) -> np.ndarray:
    """(q - zero) * scale in float64 for canonical arrays [..., rows, *]."""
    q = unpack(codes, K, wbits).astype(np.float64)
    s = np.asarray(scales, np.uint16).view(np.float16).astype(np.float64)
    z = np.asarray(zeros, np.uint8).astype(np.float64)
    s = np.repeat(s, group, axis=-1)
    z = np.repeat(z, group, axis=-1)
    return (q - z) * s


def f16(bits) -> np.ndarray:
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def half_fraction(b: int) -> Fraction:
    return Fraction(float(np.array(b, np.uint16).view(np.float16)))


def f32_round(fr: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) float32 of a rational in the
    normal range."""
    if fr == 0:
        return np.float32(0.0)
    neg = fr < 0
    a = -fr if neg else fr
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while a >= Fraction(2) ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    assert -126 <= e <= 127
    q = a / Fraction(2) ** (e - 23)       # in [2^23, 2^24)
    m = q.numerator // q.denominator
    rem = q - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    if m == 1 << 24:
        m >>= 1
        e += 1
    bits = (int(neg) << 31) | ((e + 127) << 23) | (m - (1 << 23))
    return np.array(bits, np.uint32).view(np.float32)[()]


def exact_logits(x_bits, rw_bits, bias=None) -> np.ndarray:
    """Router logits from exact rational dot products, rounded once to fp32,
    then one float32 add of the bias."""
    x_bits = np.asarray(x_bits, np.uint16)
    rw_bits = np.asarray(rw_bits, np.uint16)
    xf = [[half_fraction(b) for b in row] for row in x_bits]
    wf = [[half_fraction(b) for b in row] for row in rw_bits]
    n, E = len(xf), len(wf)
    out = np.empty((n, E), np.float32)
    for t in range(n):
        for e in range(E):
            l = f32_round(sum((a * b for a, b in zip(xf[t], wf[e])), Fraction(0)))
            if bias is not None:
                l = np.float32(l) + np.float32(bias[e])
            out[t, e] = l
    return out


def topk_ref(logits: np.ndarray, k: int):
    """Stable descending sort (ties keep the lower expert id); softmax over the
    selected logits in float64."""
    n, E = logits.shape
    idx = np.empty((n, k), np.int64)
    w = np.empty((n, k), np.float64)
    for t in range(n):
        order = sorted(range(E), key=lambda e: -float(logits[t, e]))  # sorted() is stable
        sel = order[:k]
        idx[t] = sel
        v = np.array([float(logits[t, e]) for e in sel])
        ex = np.exp(v - v.max())
        w[t] = ex / ex.sum()
    return idx, w


def silu(v):
    return v / (1.0 + np.exp(-v))


def dense_ffn(layer, e, x):
    """y = W_down (silu(W_gate x) * (W_up x)) with numpy matmuls; e = -1 for
    the shared expert.  x: float64 [T, H]."""
    s = layer.spec
    if e < 0:
        I = s.shared_inter
        c, sc, z = layer.sh_codes, layer.sh_scales, layer.sh_zeros
        e = 0
    else:
        I = s.inter
        c, sc, z = layer.codes, layer.scales, layer.zeros
    Wg = dequant(c[0][e], sc[0][e], z[0][e], s.hidden, s.wbits, s.group)
    Wu = dequant(c[1][e], sc[1][e], z[1][e], s.hidden, s.wbits, s.group)
    Wd = dequant(c[2][e], sc[2][e], z[2][e], I, s.wbits, s.group)
    g = x @ Wg.T
    u = x @ Wu.T
    return (silu(g) * u) @ Wd.T
