"""ctypes wrapper around the C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of the
benchmark).  Arguments are numpy arrays in the canonical packed format; fp16
values travel as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import hashlib
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_lib", "liboracle.so")
_lib = None


def _source_hash(paths, flags) -> str:
    h = hashlib.sha256(" ".join(flags).encode())
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (fp contraction off, no fast-math, OpenMP).
    Rebuilds whenever the sources or flags differ from those of the library
    on disk (a hash of both is kept beside it)."""
    src = os.path.join(_HERE, "oracle.c")
    hdr = os.path.join(_HERE, "oracle.h")
    flags = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
             "-shared", "-Wall"]
    digest = _source_hash([src, hdr], flags)
    stamp = _SO + ".sha256"
    if (not force and os.path.exists(_SO) and os.path.exists(stamp)
            and open(stamp).read().strip() == digest):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *flags, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, _SO)
    with open(stamp, "w") as f:
        f.write(digest + "\n")
    return _SO


class OracleLayer(C.Structure):
    _fields_ = [
        ("hidden", C.c_int), ("inter", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
        ("group", C.c_int), ("wbits", C.c_int), ("has_shared", C.c_int), ("shared_inter", C.c_int),
        ("codes", C.c_void_p * 3), ("scales", C.c_void_p * 3), ("zeros", C.c_void_p * 3),
        ("router_w", C.c_void_p), ("router_bias", C.c_void_p),
        ("sh_codes", C.c_void_p * 3), ("sh_scales", C.c_void_p * 3), ("sh_zeros", C.c_void_p * 3),
        ("sh_gate_w", C.c_void_p),
    ]


def load():
    global _lib
    if _lib is None:
        so = os.environ.get("QEFFN_ORACLE_SO")   # a planted-mistake copy, from the tests
        if not so:
            so = build()
        lib = C.CDLL(so)
        P = C.c_void_p
        lib.oracle_half_to_double.restype = C.c_double
        lib.oracle_half_to_double.argtypes = [C.c_uint16]
        lib.oracle_double_to_half.restype = C.c_uint16
        lib.oracle_double_to_half.argtypes = [C.c_double]
        lib.oracle_unpack_codes.argtypes = [P, C.c_int64, C.c_int, C.c_int, P]
        lib.oracle_dequant.argtypes = [P, P, P, C.c_int64, C.c_int, C.c_int, C.c_int, P]
        lib.oracle_router_logits.argtypes = [P, C.c_int, C.c_int, P, P, C.c_int, P]
        lib.oracle_topk.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P]
        lib.oracle_group.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P]
        lib.oracle_expert_ffn.argtypes = [C.POINTER(OracleLayer), C.c_int, P, C.c_int, P]
        lib.oracle_forward.argtypes = [C.POINTER(OracleLayer), P, C.c_int, P, C.c_int,
                                       P, P, P, P, P, P, P, P]
        lib.oracle_rmsnorm.argtypes = [P, P, C.c_float, C.c_int, C.c_int, P]
        lib.oracle_num_threads.restype = C.c_int
        lib.oracle_set_num_threads.argtypes = [C.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s failed (status %d)" % (what, rc))


def half_to_double(h: int) -> float:
    return load().oracle_half_to_double(int(h))


def double_to_half(v: float) -> int:
    return int(load().oracle_double_to_half(float(v)))


def unpack_codes(codes, rows: int, K: int, wbits: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    q = np.empty((rows, K), np.uint8)
    _check(load().oracle_unpack_codes(_p(codes), rows, K, wbits, _p(q)), "unpack")
    return q


def dequant(codes, scales, zeros, rows: int, K: int, wbits: int, group: int = 128):
    codes, scales, zeros = _c(codes, np.uint8), _c(scales, np.uint16), _c(zeros, np.uint8)
    w = np.empty((rows, K), np.float64)
    _check(load().oracle_dequant(_p(codes), _p(scales), _p(zeros), rows, K, wbits, group, _p(w)),
           "dequant")
    return w


def router_logits(x, router_w, bias=None) -> np.ndarray:
    x, rw = _c(x, np.uint16), _c(router_w, np.uint16)
    n, H = x.shape
    E = rw.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((n, E), np.float32)
    _check(load().oracle_router_logits(_p(x), n, H, _p(rw), _p(b), E, _p(out)), "router")
    return out


def topk(logits, k: int):
    lg = _c(logits, np.float32)
    n, E = lg.shape
    idx = np.empty((n, k), np.int32)
    w32 = np.empty((n, k), np.float32)
    w64 = np.empty((n, k), np.float64)
    _check(load().oracle_topk(_p(lg), n, E, k, _p(idx), _p(w32), _p(w64)), "topk")
    return idx, w32, w64


def group(idx, n_experts: int):
    idx = _c(idx, np.int32)
    n, k = idx.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(n * k, np.int32)
    _check(load().oracle_group(_p(idx), n, k, n_experts, _p(counts), _p(offsets), _p(perm)),
           "group")
    return counts, offsets, perm


def _layer_struct(layer):
    """OracleLayer view of a synth.PackedLayer (keeps references alive)."""
    s = layer.spec
    keep = []

    def ptr(a, dt):
        if a is None:
            return None
        a = _c(a, dt)
        keep.append(a)
        return a.ctypes.data

    L = OracleLayer()
    L.hidden, L.inter, L.n_experts, L.top_k = s.hidden, s.inter, s.n_experts, s.top_k
    L.group, L.wbits = s.group, s.wbits
    L.has_shared, L.shared_inter = int(s.has_shared), s.shared_inter
    for m in range(3):
        L.codes[m] = ptr(layer.codes[m], np.uint8)
        L.scales[m] = ptr(layer.scales[m], np.uint16)
        L.zeros[m] = ptr(layer.zeros[m], np.uint8)
        if s.has_shared:
            L.sh_codes[m] = ptr(layer.sh_codes[m], np.uint8)
            L.sh_scales[m] = ptr(layer.sh_scales[m], np.uint16)
            L.sh_zeros[m] = ptr(layer.sh_zeros[m], np.uint8)
    L.router_w = ptr(layer.router_w, np.uint16)
    L.router_bias = ptr(layer.router_bias, np.float32)
    L.sh_gate_w = ptr(layer.sh_gate_w, np.uint16) if s.has_shared else None
    return L, keep


def expert_ffn(layer, e: int, x) -> np.ndarray:
    """y [T, H] (fp64) of expert e (-1: the shared expert) on fp16 tokens x [T, H]."""
    L, keep = _layer_struct(layer)
    x = _c(x, np.uint16)
    y = np.empty((x.shape[0], layer.spec.hidden), np.float64)
    _check(load().oracle_expert_ffn(C.byref(L), e, _p(x), x.shape[0], _p(y)), "expert_ffn")
    return y


def forward(layer, x, tokens=None, want_out=True) -> dict:
    """Route every token of x [n, H] (fp16 bits) and, for the selected tokens
    (all when tokens is None), compute the layer output.  Returns a dict with
    logits, idx, w, counts, offsets, perm and out64/out16 [n_sel, H]."""
    s = layer.spec
    L, keep = _layer_struct(layer)
    x = _c(x, np.uint16)
    n = x.shape[0]
    sel = None if tokens is None else _c(tokens, np.int32)
    ns = n if sel is None else len(sel)
    r = dict(
        logits=np.empty((n, s.n_experts), np.float32),
        idx=np.empty((n, s.top_k), np.int32),
        w=np.empty((n, s.top_k), np.float32),
        counts=np.empty(s.n_experts, np.int32),
        offsets=np.empty(s.n_experts + 1, np.int32),
        perm=np.empty(n * s.top_k, np.int32),
    )
    if want_out:
        r["out64"] = np.empty((ns, s.hidden), np.float64)
        r["out16"] = np.empty((ns, s.hidden), np.uint16)
    _check(load().oracle_forward(
        C.byref(L), _p(x), n, _p(sel), ns if want_out else 0, _p(r["logits"]), _p(r["idx"]),
        _p(r["w"]), _p(r["counts"]), _p(r["offsets"]), _p(r["perm"]),
        _p(r.get("out64")), _p(r.get("out16"))), "forward")
    return r


def rmsnorm(resid, gamma, eps: float):
    """Two-pass RMSNorm of resid [n, H] (fp16 bits) with gain gamma [H]:
    fp16 bits [n, H]."""
    r, g = _c(resid, np.uint16), _c(gamma, np.uint16)
    n, H = r.shape
    xn = np.empty((n, H), np.uint16)
    _check(load().oracle_rmsnorm(_p(r), _p(g), float(eps), n, H, _p(xn)), "rmsnorm")
    return xn


def num_threads() -> int:
    return int(load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads of the oracle's parallel loops (for single-core timing)."""
    load().oracle_set_num_threads(int(n))
