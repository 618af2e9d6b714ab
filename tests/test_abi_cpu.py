"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/moe_layer.h declares, and argument errors come back as status
codes before any CUDA call is made."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_expert_ffn_warp_gb300 import build, moe
    build.build()
    return moe.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe_layer.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    from quantized_expert_ffn_warp_gb300 import moe
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTS) == names


def _cfg(**kw):
    from quantized_expert_ffn_warp_gb300.moe import Cfg
    c = Cfg()
    d = dict(hidden=256, inter=512, n_experts=8, top_k=2, group_size=128, wbits=4, has_shared=0,
             shared_inter=0, residual=1, io_dtype=0, max_tokens=16)
    d.update(kw)
    for k, v in d.items():
        setattr(c, k, v)
    return c


def _create(lib, cfg, w):
    from quantized_expert_ffn_warp_gb300.moe import PackedWeights
    h = C.c_void_p(123)
    rc = lib.moe_layer_create(C.byref(cfg) if cfg is not None else None,
                              C.byref(w) if w is not None else None, C.byref(h))
    return rc, h.value, lib.moe_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(wbits=3), -2), (dict(wbits=8), -2), (dict(group_size=64), -2), (dict(io_dtype=1), -2),
    (dict(hidden=100), -1), (dict(hidden=0), -1), (dict(inter=130), -1),
    (dict(n_experts=0), -1), (dict(n_experts=2000), -1), (dict(top_k=0), -1),
    (dict(top_k=9), -1), (dict(top_k=33, n_experts=64), -1), (dict(max_tokens=0), -1),
    (dict(has_shared=1, shared_inter=0), -1), (dict(residual=2), -1),
])
def test_create_rejects_bad_config(lib, kw, code):
    from quantized_expert_ffn_warp_gb300.moe import PackedWeights
    rc, h, msg = _create(lib, _cfg(**kw), PackedWeights())
    assert rc == code and h is None and msg


def test_create_rejects_null_arguments(lib):
    from quantized_expert_ffn_warp_gb300.moe import PackedWeights
    assert _create(lib, None, PackedWeights())[0] == -1
    assert _create(lib, _cfg(), None)[0] == -1
    rc, h, msg = _create(lib, _cfg(), PackedWeights())      # valid cfg, null weights
    assert rc == -1 and "null" in msg
    assert lib.moe_layer_create(C.byref(_cfg()), C.byref(PackedWeights()), None) == -1


def test_calls_on_null_layer(lib):
    P = C.c_void_p
    x = P(0x1000)
    assert lib.moe_forward(None, x, P(0x2000), 1, None) == -1
    assert lib.moe_forward_routed(None, x, x, x, P(0x2000), 1, None) == -1
    assert lib.moe_route_topk(None, x, 1, None, None, None, None, None, None) == -1
    assert lib.moe_router_logits(None, x, 1, x, None) == -1
    assert lib.moe_check_status(None, None) == -1
    assert lib.moe_layer_info(None, None) == -1
    assert lib.moe_profile_enable(None, 1) == -1
    assert lib.moe_profile_read(None, None, 0, None) == -1
    assert lib.moe_forward_prenorm(None, x, x, C.c_float(1e-6), P(0x2000), 1, None) == -1
    lib.moe_layer_destroy(None)   # NULL-safe
    assert "null" in lib.moe_last_error().decode()


@pytest.mark.parametrize("args", [
    dict(resid=None), dict(xn=None), dict(gamma=None), dict(resid=0x1008), dict(gamma=0x2004),
    dict(n=0), dict(hidden=100), dict(hidden=32768), dict(eps=-1.0), dict(eps=float("nan")),
    dict(eps=float("inf")),
])
def test_rmsnorm_rejects_bad_arguments(lib, args):
    """Argument errors of the layer-free RMSNorm come back before any CUDA
    call (the pointers here are never dereferenced)."""
    a = dict(resid=0x1000, gamma=0x2000, eps=1e-6, n=4, hidden=256, xn=0x3000)
    a.update(args)
    P = C.c_void_p
    rc = lib.moe_rmsnorm(P(a["resid"]), P(a["gamma"]), C.c_float(a["eps"]), a["n"],
                         a["hidden"], P(a["xn"]), None)
    assert rc == -1 and lib.moe_last_error().decode()


def test_copy_rejects_bad_arguments(lib):
    """moe_copy: null, misaligned and overlapping ranges come back as
    INVALID_ARG before any CUDA call; zero bytes is a no-op."""
    P = C.c_void_p
    assert lib.moe_copy(P(0x1000), P(0x2000), C.c_size_t(0), None) == 0
    assert lib.moe_copy(None, P(0x2000), C.c_size_t(64), None) == -1
    assert lib.moe_copy(P(0x1000), None, C.c_size_t(64), None) == -1
    assert lib.moe_copy(P(0x1008), P(0x2000), C.c_size_t(64), None) == -1
    assert lib.moe_copy(P(0x1000), P(0x2000), C.c_size_t(40), None) == -1
    assert lib.moe_copy(P(0x1000), P(0x1010), C.c_size_t(64), None) == -1
    assert "overlap" in lib.moe_last_error().decode()
