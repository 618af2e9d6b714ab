"""Expert residency tiers on the GPU (moe_layer_set_residency): hot experts
resident in device memory, the rest in pinned host memory with a bounded
pool of device slots.  The forward of a tiered layer must give the bits of
the same layer untiered (same kernels, same records, other addresses) and
match the oracle; the slot hits, misses and contents must follow the
documented policy (misses in expert order take the least recently used free
slots, ties to the lower slot), simulated here in Python from the touched
experts of every call."""
import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth
import parity

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


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.float16)).cuda()


def simulate(touched_calls, E, resident, S):
    """The slot policy, call by call: (hits, misses, slot contents)."""
    res = set(int(e) for e in resident)
    slot_of = {}
    slot_expert, used = [-1] * S, [0] * S
    hits = misses = 0
    for call, touched in enumerate(touched_calls, 1):
        miss = []
        for e in sorted(touched):
            if e in res:
                continue
            s = slot_of.get(e, -1)
            if s >= 0:
                used[s] = call
                hits += 1
            else:
                miss.append(e)
        misses += len(miss)
        free = sorted((s for s in range(S) if used[s] != call), key=lambda s: (used[s], s))
        assert len(free) >= len(miss)
        for r, e in enumerate(miss):
            s = free[r]
            if slot_expert[s] >= 0:
                del slot_of[slot_expert[s]]
            slot_expert[s] = e
            slot_of[e] = s
            used[s] = call
    return hits, misses, slot_expert


def calibrate(moe, layer, spec, n, batches, seed):
    counts = np.zeros(spec.n_experts, np.int64)
    for b in range(batches):
        r = layer.route_topk(dev(synth.make_tokens(spec, n, seed=seed, batch=b)))
        counts += r["counts"].cpu().numpy()
    return counts


def run_tiered(moe, spec, n, frac, calls=10, gemm_min=None, max_tokens=None, check_oracle=True):
    import oracle
    packed = synth.make_layer(spec, seed=6)
    layer = moe.MoeLayer.from_packed(packed, max_tokens=max_tokens or n)
    try:
        if gemm_min is not None:
            layer.set_gemm_min_tokens(gemm_min)
        xs = [synth.make_tokens(spec, n, seed=8, batch=b) for b in range(calls)]
        base, touched = [], []
        for x in xs:
            r = layer.route_topk(dev(x))
            touched.append(set(np.nonzero(r["counts"].cpu().numpy())[0].tolist()))
            base.append(layer.forward(dev(x)).cpu().numpy().view(np.uint16))
        counts = calibrate(moe, layer, spec, n, 8, seed=9)
        R = int(round(frac * spec.n_experts))
        resident = moe.residency_plan(counts, R)
        E = spec.n_experts
        S = min(E - R, layer.cfg.max_tokens * spec.top_k)
        info0 = layer.info()
        layer.set_residency(resident, S)
        info1 = layer.info()
        # device memory: the resident experts, the slots and one zero block
        # instead of every expert
        assert info1["weight_bytes"] < info0["weight_bytes"] or R + S >= E - 1
        for i, x in enumerate(xs):
            got = layer.forward(dev(x)).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, base[i]), "call %d differs from the untiered layer" % i
        if check_oracle:
            ref = oracle.forward(packed, xs[-1])
            parity.assert_close(got, ref["out64"], "%s tiered n=%d" % (spec.name, n))
        st = layer.tier_stats()
        h, m, slots = simulate(touched, E, resident, S)
        assert (st["hits"], st["misses"]) == (h, m)
        assert list(layer.tier_slots(S)) == slots
        assert layer.check_status() == 0
        return layer, xs, base, resident, S
    except Exception:
        layer.close()
        raise


@pytest.mark.parametrize("name,n,frac", [("e64_top2_zipf", 8, 0.5), ("e64_top2_zipf", 1, 0.3),
                                         ("e512_top4_shared_2bit", 4, 0.25),
                                         ("e256_top8_shared", 16, 0.6)])
def test_tiered_forward_bit_identical(moe, name, n, frac):
    layer, *_ = run_tiered(moe, synth.CONFIGS[name], n, frac)
    layer.close()


def test_tiered_gemm_path_and_retier(moe):
    """Every expert on the tcgen05 GEMM path through the slots; then new
    tiers (every expert cold, the minimum pool) on the same layer."""
    spec = synth.CONFIGS["tiny"]
    layer, xs, base, _, _ = run_tiered(moe, spec, 37, 0.25, gemm_min=1, max_tokens=37)
    try:
        layer.set_residency([], min(spec.n_experts, 37 * spec.top_k))
        for i, x in enumerate(xs):
            assert np.array_equal(layer.forward(dev(x)).cpu().numpy().view(np.uint16), base[i])
        layer.set_residency(list(range(spec.n_experts)), 0)   # everything resident again
        assert np.array_equal(layer.forward(dev(xs[0])).cpu().numpy().view(np.uint16), base[0])
        assert layer.check_status() == 0
    finally:
        layer.close()


def test_tiered_forward_in_cuda_graph(moe):
    """The staging kernels run in the stream: a captured forward replays the
    slot decisions on the device."""
    spec = synth.CONFIGS["e64_top2_zipf"]
    layer, xs, base, _, _ = run_tiered(moe, spec, 8, 0.25, calls=4, check_oracle=False)
    try:
        st = torch.cuda.Stream()
        xd = [dev(x) for x in xs]
        outs = [torch.empty_like(xd[0]) for _ in xs]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            layer.forward(xd[0], outs[0], stream=st)    # warm
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                for i in range(len(xs)):
                    layer.forward(xd[i], outs[i], stream=st)
        for _ in range(3):
            g.replay()
            torch.cuda.synchronize()
            for i in range(len(xs)):
                assert np.array_equal(outs[i].cpu().numpy().view(np.uint16), base[i])
        assert layer.check_status() == 0
    finally:
        layer.close()


def test_set_residency_argument_errors(moe):
    spec = synth.CONFIGS["tiny"]
    layer = moe.MoeLayer.from_packed(synth.make_layer(spec), max_tokens=2)
    try:
        for resident, S in [([0, 0], 4), ([8], 4), ([-1], 4), ([0, 1], 3), ([0, 1], 7)]:
            with pytest.raises(moe.MoeError):
                layer.set_residency(resident, S)
        with pytest.raises(moe.MoeError):
            layer.tier_stats()
    finally:
        layer.close()
