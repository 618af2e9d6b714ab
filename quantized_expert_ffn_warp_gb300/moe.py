"""Thin Python binding of the C ABI in include/moe_layer.h.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe_layer.so.  PyTorch provides device memory and streams.  There is no
fallback: if the library is missing the import of a layer fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_layer.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_OOM = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_STATUS = -5
MOE_STATUS_BAD_EXPERT = 1
MOE_STATUS_NONFINITE = 2
MOE_STATUS_TIMEOUT = 4
MOE_STATUS_TIER_OVERFLOW = 8
MOE_NOALLOC_MAX_SCORES = 16384
PHASES = ("route", "group", "gate_up", "down", "combine")

EXPORTS = ("moe_layer_create", "moe_layer_destroy", "moe_route_topk", "moe_router_logits",
           "moe_forward", "moe_forward_routed", "moe_check_status", "moe_layer_info",
           "moe_profile_enable", "moe_profile_read", "moe_last_error",
           "moe_route_topk_noalloc", "moe_layer_set_gemm_min_tokens", "moe_rmsnorm",
           "moe_forward_prenorm", "moe_copy", "moe_layer_set_residency", "moe_residency_plan",
           "moe_layer_tier_stats", "moe_layer_tier_slots", "moe_ep_dispatch", "moe_ep_combine")


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("moe status %d: %s" % (code, msg))
        self.code = code


class Cfg(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("hidden", "inter", "n_experts", "top_k", "group_size",
                                        "wbits", "has_shared", "shared_inter", "residual",
                                        "io_dtype", "max_tokens")]


class PackedWeights(C.Structure):
    _fields_ = [("codes", C.c_void_p * 3), ("scales", C.c_void_p * 3), ("zeros", C.c_void_p * 3),
                ("router_w", C.c_void_p), ("router_bias", C.c_void_p),
                ("sh_codes", C.c_void_p * 3), ("sh_scales", C.c_void_p * 3),
                ("sh_zeros", C.c_void_p * 3), ("sh_gate_w", C.c_void_p)]


class LayerInfo(C.Structure):
    _fields_ = [("weight_bytes", C.c_int64), ("workspace_bytes", C.c_int64),
                ("expert_bytes", C.c_int64), ("shared_bytes", C.c_int64),
                ("num_sms", C.c_int), ("grid_ffn", C.c_int), ("n_phases", C.c_int),
                ("gemm_min_tokens", C.c_int)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libmoe_layer.so (build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libmoe_layer.so not built (%s): run __graft_entry__.build()" % path)
    lib = C.CDLL(path)
    P, I = C.c_void_p, C.c_int
    lib.moe_layer_create.argtypes = [C.POINTER(Cfg), C.POINTER(PackedWeights), C.POINTER(P)]
    lib.moe_layer_destroy.argtypes = [P]
    lib.moe_layer_destroy.restype = None
    lib.moe_route_topk.argtypes = [P, P, I, P, P, P, P, P, P]
    lib.moe_router_logits.argtypes = [P, P, I, P, P]
    lib.moe_forward.argtypes = [P, P, P, I, P]
    lib.moe_forward_routed.argtypes = [P, P, P, P, P, I, P]
    lib.moe_check_status.argtypes = [P, C.POINTER(I)]
    lib.moe_layer_info.argtypes = [P, C.POINTER(LayerInfo)]
    lib.moe_profile_enable.argtypes = [P, I]
    lib.moe_profile_read.argtypes = [P, C.POINTER(C.c_float), I, C.POINTER(I)]
    lib.moe_layer_set_gemm_min_tokens.argtypes = [P, I]
    lib.moe_route_topk_noalloc.argtypes = [P, P, P, I, I, I, I, P, P, P]
    lib.moe_rmsnorm.argtypes = [P, P, C.c_float, I, I, P, P]
    lib.moe_forward_prenorm.argtypes = [P, P, P, C.c_float, P, I, P]
    lib.moe_copy.argtypes = [P, P, C.c_size_t, P]
    lib.moe_layer_set_residency.argtypes = [P, P, I, I]
    lib.moe_residency_plan.argtypes = [P, I, I, P]
    lib.moe_layer_tier_stats.argtypes = [P, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64),
                                         C.POINTER(I)]
    lib.moe_layer_tier_slots.argtypes = [P, P, I]
    lib.moe_ep_dispatch.argtypes = [P, I, I, P, I, I, I, P, P, P, P, P, P]
    lib.moe_ep_combine.argtypes = [P, I, I, I, P, P, P, P, P, I, P, P]
    lib.moe_last_error.restype = C.c_char_p
    lib.moe_last_error.argtypes = []
    _lib = lib
    return lib


def _check(rc):
    if rc != MOE_OK:
        raise MoeError(rc, load_library().moe_last_error().decode())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def make_cfg(spec, max_tokens=None, residual=1) -> Cfg:
    c = Cfg()
    c.hidden, c.inter, c.n_experts, c.top_k = spec.hidden, spec.inter, spec.n_experts, spec.top_k
    c.group_size, c.wbits = spec.group, spec.wbits
    c.has_shared, c.shared_inter = int(spec.has_shared), spec.shared_inter
    c.residual, c.io_dtype = residual, 0
    c.max_tokens = spec.max_tokens if max_tokens is None else max_tokens
    return c


def upload(layer, device="cuda"):
    """Device copies (torch tensors) of a synth.PackedLayer's canonical buffers."""
    import torch

    def t(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:      # fp16 bit patterns travel as int16
            a = a.view(np.int16)
        return torch.from_numpy(a).to(device)

    d = dict(codes=[t(a) for a in layer.codes], scales=[t(a) for a in layer.scales],
             zeros=[t(a) for a in layer.zeros], router_w=t(layer.router_w),
             router_bias=t(layer.router_bias))
    if layer.spec.has_shared:
        d.update(sh_codes=[t(a) for a in layer.sh_codes], sh_scales=[t(a) for a in layer.sh_scales],
                 sh_zeros=[t(a) for a in layer.sh_zeros], sh_gate_w=t(layer.sh_gate_w))
    return d


def route_topk_noalloc(x, router_w, router_bias, top_k, stream=None, idx=None, w=None):
    """Routing (top-k ids and softmax weights) of x fp16 [n, H] against
    router_w fp16 [E, H] (+ router_bias fp32 [E] or None) through
    moe_route_topk_noalloc: no layer object, no device allocation inside the
    library.  Returns (idx int32 [n, k], w fp32 [n, k]), written into the
    given contiguous tensors when idx and w are passed."""
    import torch
    n, H = x.shape
    E = router_w.shape[0]
    if idx is None:
        idx = torch.empty((n, top_k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((n, top_k), dtype=torch.float32, device=x.device)
    _check(load_library().moe_route_topk_noalloc(_ptr(x), _ptr(router_w), _ptr(router_bias), n, H,
                                                 E, top_k, _ptr(idx), _ptr(w), _stream(stream)))
    return idx, w


class MoeLayer:
    """One quantised MoE layer owned by libmoe_layer.so."""

    def __init__(self, spec, weights: dict, max_tokens=None, residual=1):
        lib = load_library()
        self.spec = spec
        self.cfg = make_cfg(spec, max_tokens, residual)
        w = PackedWeights()
        for m in range(3):
            w.codes[m] = weights["codes"][m].data_ptr()
            w.scales[m] = weights["scales"][m].data_ptr()
            w.zeros[m] = weights["zeros"][m].data_ptr()
        w.router_w = weights["router_w"].data_ptr()
        rb = weights.get("router_bias")
        w.router_bias = rb.data_ptr() if rb is not None else None
        if spec.has_shared:
            for m in range(3):
                w.sh_codes[m] = weights["sh_codes"][m].data_ptr()
                w.sh_scales[m] = weights["sh_scales"][m].data_ptr()
                w.sh_zeros[m] = weights["sh_zeros"][m].data_ptr()
            w.sh_gate_w = weights["sh_gate_w"].data_ptr()
        h = C.c_void_p()
        _check(lib.moe_layer_create(C.byref(self.cfg), C.byref(w), C.byref(h)))
        self._h = h

    @classmethod
    def from_packed(cls, layer, max_tokens=None, device="cuda"):
        w = upload(layer, device)
        obj = cls(layer.spec, w, max_tokens)
        del w   # create() synchronised: the canonical copies may go
        return obj

    # -- calls -------------------------------------------------------------
    def forward(self, x, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(x)
        _check(load_library().moe_forward(self._h, _ptr(x), _ptr(out), x.shape[0], _stream(stream)))
        return out

    def forward_prenorm(self, resid, gamma, eps, out=None, stream=None):
        """The layer on rmsnorm(resid, gamma, eps), with resid as its residual."""
        import torch
        if out is None:
            out = torch.empty_like(resid)
        _check(load_library().moe_forward_prenorm(self._h, _ptr(resid), _ptr(gamma), float(eps),
                                                  _ptr(out), resid.shape[0], _stream(stream)))
        return out

    def forward_routed(self, x, topk_idx, topk_w, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(x)
        _check(load_library().moe_forward_routed(self._h, _ptr(x), _ptr(topk_idx), _ptr(topk_w),
                                                 _ptr(out), x.shape[0], _stream(stream)))
        return out

    def route_topk(self, x, stream=None):
        import torch
        n, k, E = x.shape[0], self.spec.top_k, self.spec.n_experts
        dev = x.device
        r = dict(idx=torch.empty((n, k), dtype=torch.int32, device=dev),
                 w=torch.empty((n, k), dtype=torch.float32, device=dev),
                 counts=torch.empty(E, dtype=torch.int32, device=dev),
                 offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                 perm=torch.empty(n * k, dtype=torch.int32, device=dev))
        _check(load_library().moe_route_topk(self._h, _ptr(x), n, _ptr(r["idx"]), _ptr(r["w"]),
                                             _ptr(r["counts"]), _ptr(r["offsets"]),
                                             _ptr(r["perm"]), _stream(stream)))
        return r

    def router_logits(self, x, stream=None):
        import torch
        out = torch.empty((x.shape[0], self.spec.n_experts), dtype=torch.float32, device=x.device)
        _check(load_library().moe_router_logits(self._h, _ptr(x), x.shape[0], _ptr(out),
                                                _stream(stream)))
        return out

    def check_status(self):
        bits = C.c_int(0)
        rc = load_library().moe_check_status(self._h, C.byref(bits))
        if rc not in (MOE_OK, MOE_ERR_DEVICE_STATUS):
            _check(rc)
        return bits.value

    def info(self) -> dict:
        i = LayerInfo()
        _check(load_library().moe_layer_info(self._h, C.byref(i)))
        return {f: getattr(i, f) for f, _ in LayerInfo._fields_}

    def set_gemm_min_tokens(self, min_tokens):
        """Experts with at least min_tokens tokens use the tensor-core GEMM
        kernels; 0 keeps every expert on the decode kernels."""
        _check(load_library().moe_layer_set_gemm_min_tokens(self._h, int(min_tokens)))

    def set_residency(self, resident, n_slots):
        """Keep the experts in `resident` in device memory and the rest in
        pinned host memory, with n_slots device slots caching those in use."""
        r = np.ascontiguousarray(np.asarray(resident, np.int32))
        _check(load_library().moe_layer_set_residency(
            self._h, r.ctypes.data_as(C.c_void_p) if r.size else None, int(r.size), int(n_slots)))

    def tier_stats(self) -> dict:
        hits, misses, filled = C.c_uint64(0), C.c_uint64(0), C.c_int(0)
        _check(load_library().moe_layer_tier_stats(self._h, C.byref(hits), C.byref(misses),
                                                    C.byref(filled)))
        return dict(hits=hits.value, misses=misses.value, slots_filled=filled.value)

    def tier_slots(self, n_slots):
        out = np.empty(max(n_slots, 1), np.int32)
        _check(load_library().moe_layer_tier_slots(self._h, out.ctypes.data_as(C.c_void_p),
                                                   int(out.size)))
        return out[:n_slots]

    def profile_enable(self, on=True):
        _check(load_library().moe_profile_enable(self._h, int(on)))

    def profile_read(self):
        ms = (C.c_float * len(PHASES))()
        calls = C.c_int(0)
        _check(load_library().moe_profile_read(self._h, ms, len(PHASES), C.byref(calls)))
        return dict(zip(PHASES, list(ms))), calls.value

    def close(self):
        if getattr(self, "_h", None):
            load_library().moe_layer_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def residency_plan(counts, n_resident):
    """The n_resident most frequently routed experts (ties to the lower id)
    from per-expert counts, by the library's placement policy."""
    c = np.ascontiguousarray(np.asarray(counts, np.int64))
    out = np.empty(max(n_resident, 1), np.int32)
    _check(load_library().moe_residency_plan(c.ctypes.data_as(C.c_void_p), int(c.size),
                                             int(n_resident), out.ctypes.data_as(C.c_void_p)))
    return out[:n_resident]


def ep_dispatch(x, topk_idx, n_experts, world, stream=None):
    """moe_ep_dispatch: (send_x fp16 [P, H], send_expert int32 [P], pos_of_pair
    int32 [P], dest_counts int32 [world], status int32 [1]) on x's device;
    the first sum(dest_counts) rows of send_x / send_expert are the packed
    rows."""
    import torch
    n, H = x.shape
    k = topk_idx.shape[1]
    P = n * k
    dev = x.device
    send_x = torch.empty((P, H), dtype=torch.float16, device=dev)
    send_e = torch.empty(P, dtype=torch.int32, device=dev)
    pos = torch.empty(P, dtype=torch.int32, device=dev)
    counts = torch.empty(world, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(load_library().moe_ep_dispatch(_ptr(x), n, H, _ptr(topk_idx), k, int(n_experts),
                                          int(world), _ptr(send_x), _ptr(send_e), _ptr(pos),
                                          _ptr(counts), _ptr(status), _stream(stream)))
    return send_x, send_e, pos, counts, status


def ep_combine(x, topk_w, pos_of_pair, y_rows, sh_gate_w=None, y_shared=None, residual=1,
               out=None, stream=None):
    """moe_ep_combine: out fp16 [n, H] = x + sum_j w y[pos] + sigmoid(x . wg) y_sh."""
    import torch
    n, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(load_library().moe_ep_combine(_ptr(x), n, H, topk_w.shape[1], _ptr(topk_w),
                                         _ptr(pos_of_pair), _ptr(y_rows), _ptr(sh_gate_w),
                                         _ptr(y_shared), int(residual), _ptr(out),
                                         _stream(stream)))
    return out


def rmsnorm(resid, gamma, eps, out=None, stream=None):
    """Two-pass RMSNorm of resid fp16 [n, H] with gain gamma fp16 [H] through
    moe_rmsnorm (no layer): fp16 [n, H]."""
    import torch
    if out is None:
        out = torch.empty_like(resid)
    n, H = resid.shape
    _check(load_library().moe_rmsnorm(_ptr(resid), _ptr(gamma), float(eps), n, H, _ptr(out),
                                      _stream(stream)))
    return out


def copy(dst, src, stream=None):
    """dst <- src (same byte size) by the library's copy kernel (moe_copy):
    device tensors or pinned host tensors."""
    nbytes = src.numel() * src.element_size()
    assert dst.numel() * dst.element_size() == nbytes
    _check(load_library().moe_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)))
    return dst


def forward_host(layer: MoeLayer, x_host, out_host, stream=None, norm=None):
    """End-to-end call with pinned host buffers (asynchronous on `stream`; the
    caller synchronises): the host -> device copy of x by the library's copy
    kernel (moe_copy: the SMs read the pinned rows in place, chained with the
    layer's kernels), then the layer, whose last kernel writes the output
    rows straight into out_host.  The device staging buffer of x is cached
    per layer.  norm = (gamma, eps): x is a residual stream and the layer
    runs with the RMSNorm in front (moe_forward_prenorm)."""
    import torch
    n, H = x_host.shape
    st = stream if stream is not None else torch.cuda.current_stream()
    bufs = getattr(layer, "_host_bufs", None)
    if bufs is None or bufs.shape[0] < n:
        bufs = torch.empty((layer.cfg.max_tokens, H), dtype=torch.float16, device="cuda")
        layer._host_bufs = bufs
    xd = bufs[:n]
    with torch.cuda.stream(st):
        copy(xd, x_host, stream=st)
        if norm is None:
            layer.forward(xd, out_host, stream=st)
        else:
            layer.forward_prenorm(xd, norm[0], norm[1], out_host, stream=st)
    return out_host
