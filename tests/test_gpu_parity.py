"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Routing outputs (top-k indices, counts, offsets, permutation, logits) must be
bit-exact; top-k weights within 2e-6; layer outputs within the tolerance in
tests/parity.py.  Inputs come from the seeded generator; expected values are
computed by the oracle at test time on the same inputs.
"""
import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth
import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_expert_ffn_warp_gb300 import build
    import oracle
    build.build()
    oracle.build()
    from quantized_expert_ffn_warp_gb300 import moe
    moe.load_library()
    return moe


_cache = {}


def get_layer(env, spec, seed=0, max_tokens=None):
    key = (spec, seed, max_tokens)
    if key not in _cache:
        if len(_cache) >= 2:          # keep host and device memory bounded
            for v in _cache.values():
                v[1].close()
            _cache.clear()
            torch.cuda.empty_cache()
        packed = synth.make_layer(spec, seed)
        _cache[key] = (packed, env.MoeLayer.from_packed(packed, max_tokens=max_tokens))
    return _cache[key]


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.float16)).cuda()


def check_routing(layer, x, ref):
    xd = dev(x)
    r = layer.route_topk(xd)
    lg = layer.router_logits(xd)
    torch.cuda.synchronize()
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), ref["logits"].view(np.uint32))
    assert np.array_equal(r["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(r["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
    np.testing.assert_allclose(r["w"].cpu().numpy(), ref["w"], rtol=0, atol=2e-6)


def run_case(env, spec, n, seed=0, sample=None, batch=0):
    import oracle
    packed, layer = get_layer(env, spec, seed)
    x = synth.make_tokens(spec, n, seed=seed, batch=batch)
    tokens = None
    if sample is not None and sample < n:
        rng = np.random.default_rng(n)
        tokens = np.sort(rng.choice(n, size=sample, replace=False)).astype(np.int32)
    ref = oracle.forward(packed, x, tokens=tokens)
    check_routing(layer, x, ref)
    out = layer.forward(dev(x))
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    if tokens is not None:
        got = got[tokens]
    s = parity.assert_close(got, ref["out64"], "%s n=%d" % (spec.name, n))
    assert layer.check_status() == 0
    return s


SMALL = [("tiny", 4), ("tiny", 1), ("tiny", 37), ("tiny", 64),
         ("e64_top2_zipf", 8), ("e64_top2_zipf", 1), ("e64_top2_zipf", 64),
         ("e256_top8_shared", 1), ("e256_top8_shared", 16),
         ("e512_top4_shared", 1), ("e512_top4_shared", 4), ("e512_top4_shared", 32),
         ("e512_top4_shared_2bit", 1), ("e512_top4_shared_2bit", 4),
         ("e512_top4_shared_2bit", 32)]


@pytest.mark.parametrize("name,n", SMALL)
def test_config_parity(env, name, n):
    run_case(env, synth.CONFIGS[name], n)


@pytest.mark.parametrize("name", ["e64_top2_sweep", "e64_top2_sweep_zipf"])
@pytest.mark.parametrize("n", [1, 8, 64, 256, 1024])
def test_sweep_parity_sampled(env, name, n):
    """Full-size 64 x (4096 x 14336) layers: routing bit-exact for all n
    tokens, outputs on up to 6 sampled tokens."""
    run_case(env, synth.CONFIGS[name], n, sample=6)


RAGGED = synth.LayerSpec("ragged", hidden=384, inter=640, n_experts=12, top_k=3,
                         has_shared=True, shared_inter=384, zipf_s=0.8, max_tokens=40)


@pytest.mark.parametrize("wbits", [4, 2])
@pytest.mark.parametrize("n", [1, 5, 13, 37, 40])
def test_ragged_shapes(env, wbits, n):
    run_case(env, RAGGED.with_(wbits=wbits), n)


@pytest.mark.parametrize("name,n", [("tiny", 37), ("e64_top2_zipf", 64), ("e256_top8_shared", 16),
                                    ("e512_top4_shared", 32), ("ragged", 40)])
def test_decode_only_multi_entry_experts(env, name, n):
    """4-bit layers with every expert on the decode kernels: an expert with
    more than 8 tokens in the call gets several 8-token entries, each of
    which streams the expert's weights, and the shared expert one entry per
    8 tokens."""
    spec = RAGGED if name == "ragged" else synth.CONFIGS[name]
    packed, layer = get_layer(env, spec)
    m0 = layer.info()["gemm_min_tokens"]
    layer.set_gemm_min_tokens(0)
    try:
        run_case(env, spec, n)
    finally:
        layer.set_gemm_min_tokens(m0)


def test_single_expert_and_dense_mixture(env):
    run_case(env, synth.LayerSpec("e1", hidden=256, inter=256, n_experts=1, top_k=1,
                                  has_shared=True, shared_inter=128, max_tokens=20), 20)
    run_case(env, synth.LayerSpec("kE", hidden=256, inter=384, n_experts=4, top_k=4,
                                  zipf_s=0.5, max_tokens=20), 19)


def _tie_layer(spec):
    """Zero router: every logit ties, experts 0..k-1 take every token."""
    E = spec.n_experts
    rng = np.random.default_rng(9)
    q, s, z = [], [], []
    for m in range(3):
        rows, K = spec.mat_shape(m)
        q.append(rng.integers(0, 16, size=(E, rows, K)))
        s.append(rng.uniform(0.005, 0.02, size=(E, rows, K // 128)))
        z.append(rng.integers(6, 10, size=(E, rows, K // 128)))
    return synth.layer_from_codes(spec, q, s, z, np.zeros((E, spec.hidden)))


def test_ties_and_hot_expert(env):
    import oracle
    spec = synth.LayerSpec("ties", hidden=256, inter=256, n_experts=16, top_k=4, max_tokens=40)
    packed = _tie_layer(spec)
    layer = env.MoeLayer.from_packed(packed)
    x = synth.make_tokens(spec, 37)
    ref = oracle.forward(packed, x)
    assert np.all(ref["idx"] == np.arange(4))
    check_routing(layer, x, ref)
    out = layer.forward(dev(x))
    torch.cuda.synchronize()
    parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"])
    layer.close()


def test_ties_large_batch_route(env):
    """Zero router at a batch size that takes the large-batch route: every
    approximate logit ties, so every expert is a candidate and the exact
    logits decide; experts 0..k-1 with weight 1/k, as in the oracle."""
    import oracle
    spec = synth.LayerSpec("ties96", hidden=256, inter=256, n_experts=16, top_k=4, max_tokens=96)
    packed = _tie_layer(spec)
    layer = env.MoeLayer.from_packed(packed)
    x = synth.make_tokens(spec, 96)
    ref = oracle.forward(packed, x)
    r = layer.route_topk(dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(r["idx"].cpu().numpy(), ref["idx"])
    assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
    np.testing.assert_allclose(r["w"].cpu().numpy(), ref["w"], rtol=0, atol=2e-6)
    layer.close()


def test_bad_expert_index_sets_status(env):
    """Caller-given routing with an out-of-range expert id: the pair is
    skipped, the status word says so, every other pair is computed."""
    import oracle
    spec = synth.CONFIGS["tiny"]
    packed, layer = get_layer(env, spec)
    x = synth.make_tokens(spec, 6)
    ref = oracle.forward(packed, x)
    idx = ref["idx"].copy()
    w = ref["w"].copy()
    idx[2, 1] = spec.n_experts + 3
    idx[4, 0] = -1
    out = layer.forward_routed(dev(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    bits = layer.check_status()
    assert bits & env.MOE_STATUS_BAD_EXPERT
    assert layer.check_status() == 0          # cleared
    xf = x.view(np.float16).astype(np.float64)
    expect = xf.copy()
    for t in range(6):
        for j in range(spec.top_k):
            e = int(idx[t, j])
            if 0 <= e < spec.n_experts:
                expect[t] += float(w[t, j]) * oracle.expert_ffn(packed, e, x[t:t + 1])[0]
    parity.assert_close(out.cpu().numpy().view(np.uint16), expect)


def test_nonfinite_input_sets_status(env):
    """An inf in one token's hidden state: the router flags it in the status
    word (the value counts as zero in the exact logit) and the other tokens'
    routing and outputs are unchanged, bit for bit."""
    spec = synth.CONFIGS["tiny"]
    packed, layer = get_layer(env, spec)
    x = synth.make_tokens(spec, 4)
    clean = layer.forward(dev(x))
    r_clean = layer.route_topk(dev(x))
    torch.cuda.synchronize()
    assert layer.check_status() == 0
    bad = x.copy()
    bad[1, 5] = 0x7C00                        # +inf in fp16
    out = layer.forward(dev(bad))
    r_bad = layer.route_topk(dev(bad))
    torch.cuda.synchronize()
    assert layer.check_status() & env.MOE_STATUS_NONFINITE
    assert layer.check_status() == 0          # cleared
    keep = [0, 2, 3]
    assert np.array_equal(r_bad["idx"].cpu().numpy()[keep], r_clean["idx"].cpu().numpy()[keep])
    assert np.array_equal(out.cpu().numpy()[keep], clean.cpu().numpy()[keep])


def test_argument_errors(env):
    spec = synth.CONFIGS["tiny"]
    packed, layer = get_layer(env, spec)
    x = dev(synth.make_tokens(spec, 8))
    lib = env.load_library()
    import ctypes as C
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty_like(x)
    assert lib.moe_forward(layer._h, C.c_void_p(x.data_ptr()), C.c_void_p(out.data_ptr()), 0, st) == -1
    assert lib.moe_forward(layer._h, C.c_void_p(x.data_ptr()), C.c_void_p(out.data_ptr()),
                           spec.max_tokens + 1, st) == -1
    assert lib.moe_forward(layer._h, C.c_void_p(x.data_ptr()), C.c_void_p(x.data_ptr()), 8, st) == -1
    assert lib.moe_forward(layer._h, C.c_void_p(x.data_ptr() + 2), C.c_void_p(out.data_ptr()),
                           4, st) == -1
    assert lib.moe_forward(layer._h, C.c_void_p(x.data_ptr()), None, 8, st) == -1
    assert layer.check_status() == 0


def _within_one_ulp(got16, ref16, what):
    """fp16 results within one ulp of the oracle's correctly rounded fp64
    value, and equal to it in at least 99% of the entries."""
    a = np.asarray(got16).view(np.int16).astype(np.int32)
    b = np.asarray(ref16).view(np.int16).astype(np.int32)
    # ordered integer images of the fp16 patterns (negative values mirrored)
    a = np.where(a < 0, -(a & 0x7FFF), a)
    b = np.where(b < 0, -(b & 0x7FFF), b)
    ulps = np.abs(a - b)
    assert ulps.max() <= 1, "%s: %d ulps" % (what, ulps.max())
    assert (ulps == 0).mean() >= 0.99, "%s: %.4f exact" % (what, (ulps == 0).mean())


@pytest.mark.parametrize("H,n,eps", [(256, 3, 1e-6), (2048, 17, 1e-5), (4096, 8, 1e-6),
                                     (16384, 2, 1e-2)])
def test_rmsnorm_parity(env, H, n, eps):
    """The layer-free RMSNorm against the oracle's fp64 definition: within one
    fp16 ulp everywhere and exact in at least 99% of the entries (the kernel
    works in fp32 in one fixed order); in place too, and deterministic."""
    import oracle
    spec = synth.LayerSpec("norm%d" % H, hidden=H, inter=128, n_experts=2, top_k=1)
    r = synth.make_residual(spec, n, batch=n)
    g = synth.make_norm_gain(spec)
    ref = oracle.rmsnorm(r, g, eps)
    got = env.rmsnorm(dev(r), dev(g), eps)
    torch.cuda.synchronize()
    got = got.cpu().numpy().view(np.uint16)
    _within_one_ulp(got, ref, "rmsnorm H=%d" % H)
    inplace = dev(r)
    env.rmsnorm(inplace, dev(g), eps, out=inplace)
    torch.cuda.synchronize()
    assert np.array_equal(inplace.cpu().numpy().view(np.uint16), got)


@pytest.mark.parametrize("name,n,min_tokens", [("tiny", 4, None), ("e64_top2_zipf", 8, None),
                                               ("e512_top4_shared", 4, None),
                                               ("e256_top8_shared", 16, None),
                                               ("tiny", 37, 1)])
def test_forward_prenorm_parity(env, name, n, min_tokens):
    """The layer with the RMSNorm in front.  The normalised tokens the GPU
    computed are first checked against the oracle's RMSNorm (within one fp16
    ulp); the oracle layer then runs on those same tokens, so that routing
    (a decision taken on fp16 inputs) is compared bit for bit on identical
    inputs, and out = resid + MoE(xn) within the tolerance, with the residual
    taken from the un-normalised rows."""
    import oracle
    spec = synth.CONFIGS[name]
    packed, layer = get_layer(env, spec)
    m0 = layer.info()["gemm_min_tokens"]
    if min_tokens is not None:
        layer.set_gemm_min_tokens(min_tokens)
    try:
        eps = 1e-6
        r = synth.make_residual(spec, n, batch=3)
        g = synth.make_norm_gain(spec)
        xn_gpu = env.rmsnorm(dev(r), dev(g), eps)
        torch.cuda.synchronize()
        xn = xn_gpu.cpu().numpy().view(np.uint16)
        _within_one_ulp(xn, oracle.rmsnorm(r, g, eps), "%s prenorm xn" % name)
        ref = oracle.forward(packed, xn)
        rt = layer.route_topk(xn_gpu)
        out = layer.forward_prenorm(dev(r), dev(g), eps)
        torch.cuda.synchronize()
        assert np.array_equal(rt["idx"].cpu().numpy(), ref["idx"])
        assert np.array_equal(rt["perm"].cpu().numpy(), ref["perm"])
        expect = (ref["out64"] - xn.view(np.float16).astype(np.float64)
                  + r.view(np.float16).astype(np.float64))
        parity.assert_close(out.cpu().numpy().view(np.uint16), expect,
                            "%s prenorm n=%d" % (name, n))
        assert layer.check_status() == 0
    finally:
        layer.set_gemm_min_tokens(m0)


def test_copy_kernel_pinned_round_trip(env):
    """moe_copy moves rows pinned host -> device -> pinned host bit for bit
    (the SMs reach the pinned rows in place), and refuses pageable host
    memory, which the device cannot reach."""
    import ctypes as C
    src = torch.randint(-30000, 30000, (37, 256), dtype=torch.int16).pin_memory()
    dev_buf = torch.empty((37, 256), dtype=torch.int16, device="cuda")
    back = torch.zeros((37, 256), dtype=torch.int16).pin_memory()
    env.copy(dev_buf, src)
    env.copy(back, dev_buf)
    torch.cuda.synchronize()
    assert torch.equal(dev_buf.cpu(), src)
    assert torch.equal(back, src)
    pageable = np.zeros(37 * 256, np.int16)
    lib = env.load_library()
    rc = lib.moe_copy(C.c_void_p(dev_buf.data_ptr()), C.c_void_p(pageable.ctypes.data),
                      C.c_size_t(pageable.nbytes), None)
    assert rc == -1 and "pinned" in lib.moe_last_error().decode()


def test_forward_host_matches_forward(env):
    """The end-to-end call (a kernel copy of the pinned input rows; the last
    kernel writes the pinned output rows in place) gives the device forward's
    bits."""
    spec = synth.CONFIGS["e64_top2_zipf"]
    packed, layer = get_layer(env, spec)
    x = synth.make_tokens(spec, 8, batch=21)
    ref = layer.forward(dev(x))
    xh = torch.from_numpy(x.view(np.float16)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    env.forward_host(layer, xh, oh)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())


def test_forward_out_must_be_reachable(env):
    """An out buffer the device cannot reach (pageable host memory) is an
    argument error, refused before any kernel runs; pinned host memory is
    written in place."""
    import ctypes as C
    spec = synth.CONFIGS["tiny"]
    packed, layer = get_layer(env, spec)
    x = dev(synth.make_tokens(spec, 4, batch=2))
    ref = layer.forward(x)
    pageable = np.zeros((4, spec.hidden), np.float16)
    lib = env.load_library()
    rc = lib.moe_forward(layer._h, C.c_void_p(x.data_ptr()), C.c_void_p(pageable.ctypes.data), 4,
                         None)
    assert rc == env.MOE_ERR_INVALID_ARG
    assert "pinned" in lib.moe_last_error().decode()
    pinned = torch.empty((4, spec.hidden), dtype=torch.float16).pin_memory()
    layer.forward(x, pinned)
    torch.cuda.synchronize()
    assert torch.equal(pinned, ref.cpu())
    assert layer.check_status() == 0


def test_deterministic_and_stream(env):
    spec = synth.CONFIGS["e256_top8_shared"]
    packed, layer = get_layer(env, spec)
    x = dev(synth.make_tokens(spec, 16, batch=3))
    a = layer.forward(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = layer.forward(x, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_graph_capture_replays_forward(env):
    spec = synth.CONFIGS["e64_top2_zipf"]
    packed, layer = get_layer(env, spec)
    x = dev(synth.make_tokens(spec, 8, batch=5))
    out = torch.empty_like(x)
    layer.forward(x, out)
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ---- tensor-core GEMM path (experts with at least min_tokens tokens) ------

GEMM_CASES = [("tiny", 37, 1, None), ("e256_top8_shared", 16, 1, None),
              ("e512_top4_shared", 32, 2, None), ("e64_top2_zipf", 64, 8, None),
              ("e64_top2_sweep_zipf", 256, 16, 6), ("e64_top2_sweep", 1024, 24, 6)]


@pytest.mark.parametrize("name,n,min_tokens,sample", GEMM_CASES)
def test_gemm_path_parity(env, name, n, min_tokens, sample):
    """Experts with >= min_tokens tokens (and the shared expert when
    n >= min_tokens) on the tcgen05 GEMM kernels, the rest on the decode
    kernels; outputs against the oracle."""
    spec = synth.CONFIGS[name]
    packed, layer = get_layer(env, spec)
    m0 = layer.info()["gemm_min_tokens"]
    layer.set_gemm_min_tokens(min_tokens)
    try:
        run_case(env, spec, n, sample=sample, batch=2)
    finally:
        layer.set_gemm_min_tokens(m0)


def test_gemm_path_ragged_and_long_entries(env):
    """Ragged shapes (3 K-groups, 5 row tiles of 128, shared expert) with every
    expert on the GEMM path, and experts of 300 tokens (five GEMM entries of
    64 tokens, the last of 44)."""
    import oracle
    spec = RAGGED.with_(max_tokens=40)
    packed = synth.make_layer(spec, 0)
    layer = env.MoeLayer.from_packed(packed)
    layer.set_gemm_min_tokens(1)
    for n in (1, 13, 40):
        x = synth.make_tokens(spec, n)
        ref = oracle.forward(packed, x)
        out = layer.forward(dev(x))
        torch.cuda.synchronize()
        parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"], "ragged n=%d" % n)
    assert layer.check_status() == 0
    layer.close()
    spec = synth.LayerSpec("ties300", hidden=256, inter=256, n_experts=16, top_k=4,
                           max_tokens=300)
    packed = _tie_layer(spec)
    layer = env.MoeLayer.from_packed(packed)
    layer.set_gemm_min_tokens(100)
    x = synth.make_tokens(spec, 300)
    ref = oracle.forward(packed, x)
    out = layer.forward(dev(x))
    torch.cuda.synchronize()
    parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"], "ties300")
    assert layer.check_status() == 0
    layer.close()


@pytest.mark.parametrize("n,E,top_k,ties", [(300, 8, 4, True), (300, 4, 2, False),
                                            (257, 2, 1, False)])
def test_gemm_path_wide_entries(env, n, E, top_k, ties):
    """Calls averaging at least 128 tokens per expert take GEMM entries of
    128 tokens (one accumulator set): full entries, a ragged last entry
    (300 = 128 + 128 + 44 on the tied experts), the shared expert's entries,
    against the oracle."""
    import oracle
    spec = synth.LayerSpec("wide%d_%d" % (E, top_k), hidden=256, inter=384, n_experts=E,
                           top_k=top_k, has_shared=not ties, shared_inter=256, max_tokens=n)
    packed = _tie_layer(spec) if ties else synth.make_layer(spec, 5)
    layer = env.MoeLayer.from_packed(packed)
    layer.set_gemm_min_tokens(100)
    try:
        x = synth.make_tokens(spec, n, seed=n)
        ref = oracle.forward(packed, x)
        out = layer.forward(dev(x))
        torch.cuda.synchronize()
        parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"], spec.name)
        assert layer.check_status() == 0
    finally:
        layer.close()


@pytest.mark.parametrize("inter,shared_inter", [(128, 128), (256, 384), (384, 128)])
def test_gemm_path_group_counts(env, inter, shared_inter):
    """Every expert on the GEMM path with 1, 2 and 3 K-groups in the down
    projection (one step of a single group, one full step, a full step and a
    tail of one group), for the routed and the shared expert."""
    import oracle
    spec = synth.LayerSpec("groups%d_%d" % (inter, shared_inter), hidden=256, inter=inter,
                           n_experts=6, top_k=2, has_shared=True, shared_inter=shared_inter,
                           max_tokens=40)
    packed = synth.make_layer(spec, 3)
    layer = env.MoeLayer.from_packed(packed)
    layer.set_gemm_min_tokens(1)
    try:
        for n in (1, 21, 40):
            x = synth.make_tokens(spec, n, seed=n)
            ref = oracle.forward(packed, x)
            out = layer.forward(dev(x))
            torch.cuda.synchronize()
            parity.assert_close(out.cpu().numpy().view(np.uint16), ref["out64"],
                                "%s n=%d" % (spec.name, n))
        assert layer.check_status() == 0
    finally:
        layer.close()


def test_gemm_path_deterministic_and_2bit_rejected(env):
    spec = synth.CONFIGS["e256_top8_shared"]
    packed, layer = get_layer(env, spec)
    m0 = layer.info()["gemm_min_tokens"]
    layer.set_gemm_min_tokens(1)
    x = dev(synth.make_tokens(spec, 16, batch=4))
    a = layer.forward(x)
    b = layer.forward(x)
    torch.cuda.synchronize()
    layer.set_gemm_min_tokens(m0)
    assert torch.equal(a, b)
    spec2 = synth.CONFIGS["e512_top4_shared_2bit"]
    packed2, layer2 = get_layer(env, spec2)
    with pytest.raises(env.MoeError):
        layer2.set_gemm_min_tokens(1)
    layer2.set_gemm_min_tokens(0)


def test_layers_of_different_sizes_coexist(env):
    """A layer created after another with fewer experts must not shrink the
    grouping kernel's shared memory under the first one (a call of more than
    256 pairs runs the separate grouping kernel)."""
    import oracle
    big = synth.LayerSpec("coexist512", hidden=256, inter=128, n_experts=512, top_k=4,
                          max_tokens=80)
    small = synth.LayerSpec("coexist1", hidden=256, inter=128, n_experts=1, top_k=1,
                            max_tokens=4)
    pb = synth.make_layer(big, 1)
    lb = env.MoeLayer.from_packed(pb)
    ls = env.MoeLayer.from_packed(synth.make_layer(small, 1))
    try:
        x = synth.make_tokens(big, 80)
        out = lb.forward(dev(x))
        torch.cuda.synchronize()
        parity.assert_close(out.cpu().numpy().view(np.uint16), oracle.forward(pb, x)["out64"],
                            "coexist")
        assert lb.check_status() == 0
    finally:
        lb.close()
        ls.close()
