"""Seeded random layer shapes against the oracle: expert counts from 1 to
300, top-k up to 12, hidden and intermediate sizes of 1 to 12 groups of 128,
4-bit and 2-bit, with and without a shared expert and a Zipf skew, token
counts that land on both sides of the kernel-shape, fused-grouping and
large-route thresholds, and the GEMM path forced on for some of them.
Routing bit-exact, outputs within the tolerance of tests/parity.py."""
import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth
import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def shapes(count=14, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        E = int(rng.choice([1, 3, 8, 17, 64, 130, 300]))
        k = int(rng.integers(1, min(E, 12) + 1))
        wbits = int(rng.choice([4, 2]))
        shared = bool(rng.integers(0, 2))
        spec = synth.LayerSpec(
            "rand%d" % i, hidden=128 * int(rng.integers(1, 13)),
            inter=128 * int(rng.integers(1, 9)), n_experts=E, top_k=k, wbits=wbits,
            has_shared=shared, shared_inter=128 * int(rng.integers(1, 5)) if shared else 0,
            zipf_s=float(rng.choice([0.0, 0.8, 1.3])) or None, max_tokens=80)
        n = int(rng.choice([1, 2, 7, 8, 9, 16, 33, 64, 80]))
        gemm = wbits == 4 and bool(rng.integers(0, 3) == 0)
        out.append((spec, n, gemm))
    return out


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_expert_ffn_warp_gb300 import build, moe
    import oracle
    build.build()
    oracle.build()
    moe.load_library()
    return moe


@pytest.mark.parametrize("case", range(14))
def test_random_shape(env, case):
    import oracle
    spec, n, gemm = shapes()[case]
    packed = synth.make_layer(spec, seed=case)
    layer = env.MoeLayer.from_packed(packed)
    try:
        if gemm:
            layer.set_gemm_min_tokens(1)
        x = synth.make_tokens(spec, n, seed=case, batch=1)
        ref = oracle.forward(packed, x)
        xd = torch.from_numpy(x.view(np.float16)).cuda()
        r = layer.route_topk(xd)
        out = layer.forward(xd)
        torch.cuda.synchronize()
        assert np.array_equal(r["idx"].cpu().numpy(), ref["idx"])
        assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
        assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
        parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"],
                            "%s E=%d k=%d H=%d I=%d wb=%d n=%d gemm=%d" % (
                                spec.name, spec.n_experts, spec.top_k, spec.hidden, spec.inter,
                                spec.wbits, n, gemm))
        assert layer.check_status() == 0
    finally:
        layer.close()
