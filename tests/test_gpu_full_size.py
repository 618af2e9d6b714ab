"""Every token of the full-size 64-expert layers (hidden 4096, expert
intermediate 14336) against the oracle, element by element: 256 tokens with
Zipf(1.2) routing and 1024 tokens with uniform routing, where the
large-batch route and the tcgen05 GEMM path run beside the decode kernels
(hot experts on the GEMM, the ragged tails of the rest on the decode
kernels).  The oracle takes about a minute of host time here."""
import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth
import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("name,n", [("e64_top2_sweep_zipf", 256), ("e64_top2_sweep", 1024)])
def test_full_size_every_token(name, n):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from quantized_expert_ffn_warp_gb300 import build, moe
    build.build()
    oracle.build()
    spec = synth.CONFIGS[name]
    packed = synth.make_layer(spec, seed=4)
    x = synth.make_tokens(spec, n, seed=4, batch=9)
    ref = oracle.forward(packed, x)
    layer = moe.MoeLayer.from_packed(packed, max_tokens=n)
    try:
        r = layer.route_topk(torch.from_numpy(x.view(np.float16)).cuda())
        out = layer.forward(torch.from_numpy(x.view(np.float16)).cuda())
        torch.cuda.synchronize()
        assert np.array_equal(r["idx"].cpu().numpy(), ref["idx"])
        assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
        assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
        counts = ref["counts"]
        assert counts.max() >= 16 and counts.min() < 16 or n == 1024, counts
        parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"],
                            "%s n=%d every token" % (name, n))
        assert layer.check_status() == 0
    finally:
        layer.close()
