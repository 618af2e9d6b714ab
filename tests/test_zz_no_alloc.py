"""moe_route_topk_noalloc (routing on the library's fixed scratch buffer, no
layer object, no device allocation) against moe_route_topk of a layer built
from the same router weights: identical top-k ids and weights on two calls in
a row (the second call must not see anything the first left in the scratch).
Named to be collected last, so it also runs after every other GPU test."""
import ctypes as C

import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_expert_ffn_warp_gb300 import build
    build.build()
    from quantized_expert_ffn_warp_gb300 import moe as m
    m.load_library()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


WIDE = synth.LayerSpec("noalloc_h16k_k32", hidden=16384, inter=128, n_experts=64, top_k=32,
                       zipf_s=0.7, max_tokens=64)


@pytest.mark.gpu
@pytest.mark.parametrize("name,n", [("e64_top2_zipf", 8), ("e256_top8_shared", 16),
                                    ("e512_top4_shared", 32), ("tiny", 37),
                                    ("noalloc_h16k_k32", 4), ("noalloc_h16k_k32", 64)])
def test_noalloc_matches_layer_routing(moe, name, n):
    """Including the largest hidden size (16384) and top-k (32), and a call
    of 64 x 256 = 16384 scores, the buffer's limit."""
    spec = WIDE if name == WIDE.name else synth.CONFIGS[name]
    if name == WIDE.name and n == 64:
        spec = spec.with_(n_experts=256, top_k=8)
    packed = synth.make_layer(spec, seed=3)
    layer = moe.MoeLayer.from_packed(packed, max_tokens=64)
    rw = _dev(packed.router_w)
    rb = torch.from_numpy(packed.router_bias).cuda() if packed.router_bias is not None else None
    try:
        for batch in (0, 1):              # two calls in a row
            x = torch.from_numpy(synth.make_tokens(spec, n, seed=5, batch=batch).view(np.float16)).cuda()
            ref = layer.route_topk(x)
            idx, w = moe.route_topk_noalloc(x, rw, rb, spec.top_k)
            torch.cuda.synchronize()
            assert np.array_equal(idx.cpu().numpy(), ref["idx"].cpu().numpy())
            assert np.array_equal(w.cpu().numpy().view(np.uint32),
                                  ref["w"].cpu().numpy().view(np.uint32))
    finally:
        layer.close()


@pytest.mark.gpu
def test_noalloc_rejects_oversize(moe):
    lib = moe.load_library()
    x = torch.zeros((17, 1024), dtype=torch.float16, device="cuda")
    rw = torch.zeros((1024, 1024), dtype=torch.float16, device="cuda")
    idx = torch.empty((17, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((17, 2), dtype=torch.float32, device="cuda")
    rc = lib.moe_route_topk_noalloc(C.c_void_p(x.data_ptr()), C.c_void_p(rw.data_ptr()), None,
                                    17, 1024, 1024, 2, C.c_void_p(idx.data_ptr()),
                                    C.c_void_p(w.data_ptr()), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert "MOE_NOALLOC_MAX_SCORES" in lib.moe_last_error().decode()


def test_noalloc_rejects_bad_arguments_before_cuda():
    from quantized_expert_ffn_warp_gb300 import build, moe as m
    build.build()
    lib = m.load_library()
    fake = C.c_void_p(256)     # never dereferenced: the size checks come first
    assert lib.moe_route_topk_noalloc(None, fake, None, 1, 128, 8, 2, fake, fake, None) == \
        m.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk_noalloc(fake, fake, None, 17, 1024, 1024, 2, fake, fake, None) == \
        m.MOE_ERR_INVALID_ARG
    assert "MOE_NOALLOC_MAX_SCORES" in lib.moe_last_error().decode()
    for n, H, E, k in [(1, 100, 8, 2), (1, 128, 0, 1), (1, 128, 8, 9), (0, 128, 8, 2),
                       (1, 128, 2000, 2), (1, 128, 64, 33)]:
        assert lib.moe_route_topk_noalloc(fake, fake, None, n, H, E, k, fake, fake, None) == \
            m.MOE_ERR_INVALID_ARG, (n, H, E, k)
    # misaligned pointers are refused before any CUDA work (the kernel reads
    # x in 16-byte and router_w in 8-byte words): a router_w slice at an odd
    # fp16 offset, an x off its 16-byte boundary, a bias or an output off its
    # 4-byte boundary
    odd2, odd4 = C.c_void_p(258), C.c_void_p(257)
    for args in [(fake, odd2, None, fake, fake), (odd4, fake, None, fake, fake),
                 (C.c_void_p(264), fake, None, fake, fake),
                 (fake, fake, C.c_void_p(258), fake, fake), (fake, fake, None, odd2, fake),
                 (fake, fake, None, fake, odd2)]:
        xx, rw, rb, ii, ww = args
        assert lib.moe_route_topk_noalloc(xx, rw, rb, 1, 128, 8, 2, ii, ww, None) == \
            m.MOE_ERR_INVALID_ARG, args
        assert "misaligned" in lib.moe_last_error().decode()
