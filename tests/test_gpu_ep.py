"""Expert-parallel layer, GPU side, on one GPU: the ranks are emulated in
one process (their steps run one after the other; the all-to-all is a
reordering of rows on the device), so every kernel of the exchange runs
through the C ABI: routing (moe_route_topk_noalloc), moe_ep_dispatch, the
owners' expert layers (moe_forward_routed), moe_ep_combine.  The dispatch
must give the reference positions, local ids and rows bit for bit; routing
must equal the oracle's; outputs must match the oracle within the tolerance
(the result rows travel as fp16, one rounding more than the one-GPU layer)."""
import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import ep, synth
import parity
from test_ep_gloo import dispatch_reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_expert_ffn_warp_gb300 import build, moe as m
    import oracle
    build.build()
    oracle.build()
    m.load_library()
    return m


def emulate(packed, world, xs, max_rows):
    """One expert-parallel forward of every rank's tokens xs[r]."""
    backends = [ep.CudaBackend(packed, r, world, max_rows) for r in range(world)]
    try:
        E = packed.spec.n_experts
        st = []
        for r in range(world):
            x = torch.from_numpy(xs[r].view(np.float16)).cuda()
            idx, w = backends[r].route(x)
            send_x, send_e, pos, counts = backends[r].dispatch(x, idx, E, world)
            st.append(dict(x=x, idx=idx, w=w, send_x=send_x, send_e=send_e, pos=pos,
                           counts=counts, off=np.concatenate([[0], np.cumsum(counts)])))
        # owners: rows from every source, in source order
        y_recv, seg = [], []
        for o in range(world):
            parts = [(s["send_x"][s["off"][o]:s["off"][o + 1]],
                      s["send_e"][s["off"][o]:s["off"][o + 1]]) for s in st]
            rows = torch.cat([p[0] for p in parts])
            ids = torch.cat([p[1] for p in parts])
            y_recv.append(backends[o].experts(rows, ids))
            seg.append(np.concatenate([[0], np.cumsum([len(p[1]) for p in parts])]))
        outs = []
        for r, s in enumerate(st):
            back = torch.cat([y_recv[o][seg[o][r]:seg[o][r + 1]] for o in range(world)])
            outs.append(backends[r].combine(s["x"], s["w"], s["pos"], back,
                                            backends[r].shared(s["x"])))
        torch.cuda.synchronize()
        return st, outs
    finally:
        for b in backends:
            b.close()


@pytest.mark.parametrize("name,world,n", [("e64_top2_zipf", 2, 8), ("e64_top2_zipf", 4, 16),
                                          ("e512_top4_shared", 2, 4), ("ragged", 3, 13)])
def test_expert_parallel_emulated(moe, name, world, n):
    import oracle
    spec = synth.CONFIGS.get(name) or synth.LayerSpec(
        "ragged_ep", hidden=384, inter=640, n_experts=12, top_k=3, has_shared=True,
        shared_inter=384, zipf_s=0.8)
    packed = synth.make_layer(spec, seed=5)
    xs = [synth.make_tokens(spec, n + r, seed=6, batch=r) for r in range(world)]
    st, outs = emulate(packed, world, xs, max_rows=world * (n + world) * spec.top_k)
    for r in range(world):
        ref = oracle.forward(packed, xs[r])
        idx = st[r]["idx"].cpu().numpy()
        assert np.array_equal(idx, ref["idx"])
        pos, local, counts = dispatch_reference(idx, spec.n_experts, world)
        assert st[r]["counts"] == counts
        assert np.array_equal(st[r]["pos"].cpu().numpy(), pos)
        P = len(pos)
        assert np.array_equal(st[r]["send_e"].cpu().numpy()[:P], local)
        rows = st[r]["send_x"].cpu().numpy().view(np.uint16)[:P]
        assert np.array_equal(rows[pos], xs[r][np.arange(P) // spec.top_k])
        parity.assert_close(outs[r].cpu().numpy().view(np.uint16), ref["out64"],
                            "%s ep world=%d rank %d" % (name, world, r))


def test_ep_argument_errors(moe):
    lib = moe.load_library()
    import ctypes as C
    f = C.c_void_p(256)
    assert lib.moe_ep_dispatch(None, 1, 128, f, 1, 8, 2, f, f, f, f, f, None) == -1
    assert lib.moe_ep_dispatch(f, 1, 128, f, 1, 8, 40, f, f, f, f, f, None) == -1   # world
    assert lib.moe_ep_dispatch(f, 1, 100, f, 1, 8, 2, f, f, f, f, f, None) == -1    # hidden
    assert lib.moe_ep_combine(f, 1, 128, 1, f, f, f, f, None, 1, f, None) == -1     # gate only
    assert lib.moe_ep_combine(f, 1, 128, 1, f, f, f, None, None, 1, f, None) == -1  # overlap
