"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against an independent restatement
(``tests/indep.py``: numpy bit operations, exact rationals, numpy matmuls), a
closed form, an invariant, or the hand-worked case in
``tests/golden/hand_two_experts.txt``.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from quantized_expert_ffn_warp_gb300 import synth
import indep

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ fp16

def test_half_to_double_every_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_double_to_half_rne(oracle_lib):
    rng = np.random.default_rng(1)
    vals = list(rng.normal(0, 1, 2000)) + list(rng.normal(0, 3000, 2000))
    vals += list(np.exp(rng.uniform(-20, 11.2, 2000)) * rng.choice([-1, 1], 2000))
    # exact ties between adjacent halves, in normal and subnormal range, and overflow
    for b in list(range(0x0001, 0x0400, 37)) + list(range(0x0400, 0x7bff, 211)):
        lo = float(np.array(b, np.uint16).view(np.float16))
        hi = float(np.array(b + 1, np.uint16).view(np.float16))
        vals += [(lo + hi) / 2, -(lo + hi) / 2, np.nextafter((lo + hi) / 2, 0)]
    vals += [65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26,
             3 * 2.0 ** -26]
    vals = np.array(vals, np.float64)
    ref = vals.astype(np.float16).view(np.uint16)   # numpy rounds float64 -> float16 RNE
    got = np.array([oracle_lib.double_to_half(v) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# -------------------------------------------------------- unpack, dequant

@pytest.mark.parametrize("wbits", [4, 2])
def test_unpack_bruteforce(oracle_lib, wbits):
    rng = np.random.default_rng(wbits)
    rows, K = 7, 256
    q = rng.integers(0, 1 << wbits, size=(rows, K))
    codes = synth.pack_codes(q, wbits)
    assert np.array_equal(oracle_lib.unpack_codes(codes, rows, K, wbits), q)
    assert np.array_equal(indep.unpack(codes, K, wbits), q)
    # one element at a time: element k alone set to v lands where the format says
    for k in (0, 1, 2, 3, 5, 130, 255):
        for v in (1, (1 << wbits) - 1):
            qq = np.zeros((1, K), np.int64)
            qq[0, k] = v
            c = synth.pack_codes(qq, wbits)
            per = 8 // wbits
            byte, field = divmod(k, per)
            assert c[0, byte] == v << (wbits * field)
            assert np.count_nonzero(c) == 1
            assert np.array_equal(oracle_lib.unpack_codes(c, 1, K, wbits), qq)


@pytest.mark.parametrize("wbits", [4, 2])
def test_dequant_exact(oracle_lib, wbits):
    rng = np.random.default_rng(10 + wbits)
    rows, K = 5, 256
    q = rng.integers(0, 1 << wbits, size=(rows, K))
    s = rng.uniform(0.005, 0.02, size=(rows, K // 128)).astype(np.float16)
    z = rng.integers(0, 1 << wbits, size=(rows, K // 128)).astype(np.uint8)
    codes = synth.pack_codes(q, wbits)
    got = oracle_lib.dequant(codes, s.view(np.uint16), z, rows, K, wbits)
    for r in range(rows):
        for k in range(0, K, 3):
            g = k // 128
            exact = (Fraction(int(q[r, k])) - int(z[r, g])) * Fraction(float(s[r, g]))
            assert got[r, k] == float(exact)        # exactly representable: (q-z)*s
    assert np.array_equal(got, indep.dequant(codes, s.view(np.uint16), z, K, wbits))


# ---------------------------------------------------------- router logits

def _rand_half_bits(rng, shape):
    """Random finite fp16 patterns: all exponents, subnormals, both zeros."""
    b = rng.integers(0, 65536, size=shape, dtype=np.uint32).astype(np.uint16)
    inf_nan = (b & 0x7C00) == 0x7C00
    b[inf_nan] &= 0xBFFF   # clear the top exponent bit: finite
    return b


def test_router_logits_exact_random(oracle_lib):
    rng = np.random.default_rng(5)
    for trial in range(4):
        n, H, E = 3, 64 if trial < 2 else 200, 5
        if trial % 2 == 0:
            x = _rand_half_bits(rng, (n, H))
            rw = _rand_half_bits(rng, (E, H))
        else:
            x = rng.normal(0, 1, (n, H)).astype(np.float16).view(np.uint16)
            rw = rng.normal(0, 0.05, (E, H)).astype(np.float16).view(np.uint16)
        bias = rng.normal(0, 1, E).astype(np.float32)
        ref = indep.exact_logits(x, rw, bias)
        got = oracle_lib.router_logits(x, rw, bias)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        ref0 = indep.exact_logits(x, rw)
        got0 = oracle_lib.router_logits(x, rw)
        assert np.array_equal(got0.view(np.uint32), ref0.view(np.uint32))


def _h(v):
    return int(np.array(np.float16(v)).view(np.uint16))


@pytest.mark.parametrize("terms,expect", [
    # 1 + 2^-24 is a tie between 1 and 1 + 2^-23: to even -> 1
    ([(1.0, 1.0), (2.0 ** -12, 2.0 ** -12)], 1.0),
    # 1 + 3*2^-24 is a tie between 1+2^-23 and 1+2^-22: to even -> 1+2^-22
    ([(1.0, 1.0), (3 * 2.0 ** -12, 2.0 ** -12)], 1.0 + 2.0 ** -22),
    # 2^10 + 2^-14 + 2^-48: rounding through a double first would drop 2^-48
    # and land on a tie (-> 2^10); the exact sum is above the tie -> 2^10 + 2^-13
    ([(32.0, 32.0), (2.0 ** -7, 2.0 ** -7), (2.0 ** -24, 2.0 ** -24)], 1024.0 + 2.0 ** -13),
    # cancellation down to the smallest product, 2^-48
    ([(32.0, 32.0), (-32.0, 32.0), (2.0 ** -24, 2.0 ** -24)], 2.0 ** -48),
    # negative tie: -(1 + 2^-24) -> -1
    ([(-1.0, 1.0), (-(2.0 ** -12), 2.0 ** -12)], -1.0),
    # largest magnitudes: 65504^2 * 2, exact in fp32? 65504^2 = 4290774016 -> rounds
    ([(65504.0, 65504.0), (65504.0, 65504.0)], float(np.float32(2 * 65504.0 ** 2))),
])
def test_router_logits_rounding_cases(oracle_lib, terms, expect):
    x = np.array([[_h(a) for a, _ in terms]], np.uint16)
    w = np.array([[_h(b) for _, b in terms]], np.uint16)
    got = oracle_lib.router_logits(x, w)[0, 0]
    assert got == np.float32(expect)
    exact = sum((Fraction(a) * Fraction(b) for a, b in terms), Fraction(0))
    assert got == indep.f32_round(exact)


# ------------------------------------------------------------- top-k

def test_topk_ties_zero_router(oracle_lib):
    for k, E in ((2, 8), (4, 16), (8, 64)):
        idx, w32, w64 = oracle_lib.topk(np.zeros((3, E), np.float32), k)
        assert np.array_equal(idx, np.tile(np.arange(k), (3, 1)))
        assert np.all(w64 == 1.0 / k)


def test_topk_vs_stable_sort(oracle_lib):
    rng = np.random.default_rng(3)
    lg = rng.normal(0, 1, (50, 32)).astype(np.float32)
    lg[::3, 5] = lg[::3, 2]     # exact ties inside the top set
    lg[::4, 7] = lg[::4].max(axis=1)
    for k in (1, 2, 4, 8, 32):
        idx, w32, w64 = oracle_lib.topk(lg, k)
        ridx, rw = indep.topk_ref(lg, k)
        assert np.array_equal(idx, ridx)
        np.testing.assert_allclose(w64, rw, rtol=1e-15, atol=0)
        assert np.array_equal(w32, w64.astype(np.float32))
        np.testing.assert_allclose(w64.sum(axis=1), 1.0, rtol=0, atol=1e-12)


# ------------------------------------------------------------ grouping

def test_group_vs_stable_sort(oracle_lib):
    rng = np.random.default_rng(4)
    for n, k, E in ((1, 1, 1), (7, 2, 8), (33, 4, 16), (100, 8, 256)):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(n)]).astype(np.int32)
        counts, offsets, perm = oracle_lib.group(idx, E)
        flat = idx.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        ref = sorted(range(n * k), key=lambda p: flat[p])   # stable
        assert np.array_equal(perm, ref)


# ------------------------------------------------------- whole-layer cases

def _layer(spec, qd, sc, zero=8, router=None, bias=None, sh=None, gate_w=None):
    """Layer whose matrix m of expert e is constant (q - z) = qd[e][m] with
    scale sc[e][m]."""
    E = spec.n_experts
    q, s, z = [], [], []
    for m in range(3):
        rows, K = spec.mat_shape(m)
        q.append(np.stack([np.full((rows, K), zero + qd[e][m]) for e in range(E)]))
        s.append(np.stack([np.full((rows, K // 128), sc[e][m]) for e in range(E)]))
        z.append(np.full((E, rows, K // 128), zero))
    kw = {}
    if spec.has_shared:
        sq, ss, sz = [], [], []
        for m in range(3):
            rows, K = spec.mat_shape(m, shared=True)
            sq.append(np.full((1, rows, K), zero + sh[0][m]))
            ss.append(np.full((1, rows, K // 128), sh[1][m]))
            sz.append(np.full((1, rows, K // 128), zero))
        kw = dict(sh_q=sq, sh_scales=ss, sh_zeros=sz, sh_gate_w=gate_w)
    if router is None:
        router = np.zeros((E, spec.hidden))
    return synth.layer_from_codes(spec, q, s, z, router, bias, **kw)


def test_hand_worked_two_experts(oracle_lib):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "hand_two_experts.txt"))
            if l.strip() and not l.startswith("#")]
    spec = synth.LayerSpec("hand", hidden=128, inter=128, n_experts=2, top_k=2)
    router = np.stack([np.full(128, 2.0 ** -7), np.full(128, 2.0 ** -6)])
    layer = _layer(spec, qd=[[-2, 1, 3], [1, 2, -1]],
                   sc=[[2.0 ** -6, 2.0 ** -5, 2.0 ** -7], [2.0 ** -6, 2.0 ** -6, 2.0 ** -7]],
                   router=router)
    x = np.array([np.full(128, float(r[1])) for r in rows]).astype(np.float16).view(np.uint16)
    r = oracle_lib.forward(layer, x)
    _, _, w64 = oracle_lib.topk(r["logits"], 2)
    for t, row in enumerate(rows):
        assert list(r["idx"][t]) == [int(row[2]), int(row[3])]
        assert w64[t, 0] == pytest.approx(float(row[4]), rel=1e-15)
        assert w64[t, 1] == pytest.approx(float(row[5]), rel=1e-15)
        np.testing.assert_allclose(r["out64"][t], float(row[6]), rtol=1e-14)
        assert np.all(r["out16"][t] == int(row[7], 16))


def test_zero_codes_give_residual_only(oracle_lib):
    """q == zero everywhere: every expert (and the shared one) outputs 0, so
    out = fp16(x) exactly."""
    spec = synth.LayerSpec("zq", hidden=256, inter=256, n_experts=8, top_k=2, has_shared=True,
                           shared_inter=128, zipf_s=1.0)
    E = spec.n_experts
    rng = np.random.default_rng(0)
    layer = _layer(spec, qd=[[0, 0, 0]] * E, sc=[[0.01] * 3] * E,
                   router=rng.normal(0, 0.05, (E, 256)), bias=synth.zipf_bias(E, 1.0),
                   sh=([0, 0, 0], [0.01] * 3), gate_w=rng.normal(0, 0.05, 256))
    x = synth.make_tokens(spec, 9)
    r = oracle_lib.forward(layer, x)
    assert np.array_equal(r["out16"], x)


def test_constant_matrices_closed_form(oracle_lib):
    """Expert e with constant matrices a_e, b_e, d_e: g = a_e*S, u = b_e*S with
    S = sum(x), y = d_e * I * silu(g) * u in every coordinate; shared expert
    likewise behind sigmoid(x . wg)."""
    spec = synth.LayerSpec("cf", hidden=256, inter=384, n_experts=8, top_k=3, has_shared=True,
                           shared_inter=256)
    E, H, I = spec.n_experts, spec.hidden, spec.inter
    rng = np.random.default_rng(2)
    qd = [[int(rng.integers(-3, 4)), int(rng.integers(-3, 4)), int(rng.integers(-3, 4))]
          for _ in range(E)]
    sc = [[2.0 ** -8, 2.0 ** -7, 2.0 ** -9]] * E
    router = rng.normal(0, 0.05, (E, H))
    shq, shs = [2, -1, 1], [2.0 ** -8, 2.0 ** -7, 2.0 ** -9]
    gate_w = rng.normal(0, 0.05, H).astype(np.float16)
    layer = _layer(spec, qd, sc, router=router, sh=(shq, shs), gate_w=gate_w)
    x = synth.make_tokens(spec, 6)
    r = oracle_lib.forward(layer, x)
    _, _, w64 = oracle_lib.topk(r["logits"], spec.top_k)
    xf = indep.f16(x)
    for t in range(6):
        S = xf[t].sum()
        expect = xf[t].copy()
        for j in range(spec.top_k):
            e = r["idx"][t, j]
            a, b, d = (qd[e][m] * sc[e][m] for m in range(3))
            expect += w64[t, j] * d * I * (a * S / (1 + math.exp(-a * S))) * (b * S)
        a, b, d = (shq[m] * shs[m] for m in range(3))
        gate = 1 / (1 + math.exp(-(xf[t] * gate_w.astype(np.float64)).sum()))
        expect += gate * d * spec.shared_inter * (a * S / (1 + math.exp(-a * S))) * (b * S)
        np.testing.assert_allclose(r["out64"][t], expect, rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu(oracle_lib):
    """E = 1, k = 1: w = 1 and the layer is x + FFN(x) + sigmoid(x.wg) FFN_sh(x)
    for random weights (pins transposes and the gate/up order)."""
    spec = synth.LayerSpec("e1", hidden=256, inter=384, n_experts=1, top_k=1, has_shared=True,
                           shared_inter=256)
    layer = synth.make_layer(spec, seed=3)
    x = synth.make_tokens(spec, 5)
    r = oracle_lib.forward(layer, x)
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 1.0)
    xf = indep.f16(x)
    gate = 1 / (1 + np.exp(-(xf @ indep.f16(layer.sh_gate_w))))
    expect = xf + indep.dense_ffn(layer, 0, xf) + gate[:, None] * indep.dense_ffn(layer, -1, xf)
    np.testing.assert_allclose(r["out64"], expect, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(oracle_lib.expert_ffn(layer, 0, x), indep.dense_ffn(layer, 0, xf),
                               rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("wbits", [4, 2])
def test_topk_equals_all_experts_is_softmax_mixture(oracle_lib, wbits):
    """k = E: the layer is the full softmax mixture of all experts."""
    spec = synth.LayerSpec("kE", hidden=128, inter=256, n_experts=4, top_k=4, wbits=wbits,
                           zipf_s=0.7)
    layer = synth.make_layer(spec, seed=4)
    x = synth.make_tokens(spec, 3)
    r = oracle_lib.forward(layer, x)
    lg = indep.exact_logits(x, layer.router_w, layer.router_bias)
    assert np.array_equal(r["logits"].view(np.uint32), lg.view(np.uint32))
    p = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    xf = indep.f16(x)
    expect = xf.copy()
    for e in range(4):
        expect += p[:, e:e + 1] * indep.dense_ffn(layer, e, xf)
    np.testing.assert_allclose(r["out64"], expect, rtol=1e-11, atol=1e-11)


def test_routed_layer_vs_numpy(oracle_lib):
    """Tiny layer shape with k < E: out = x + sum over the selected experts of
    softmax-renormalised weight times expert output."""
    spec = synth.CONFIGS["tiny"].with_(zipf_s=0.5)
    layer = synth.make_layer(spec, seed=1)
    x = synth.make_tokens(spec, 4)
    r = oracle_lib.forward(layer, x)
    lg = indep.exact_logits(x, layer.router_w, layer.router_bias)
    idx, w = indep.topk_ref(lg, spec.top_k)
    assert np.array_equal(r["idx"], idx)
    xf = indep.f16(x)
    expect = xf.copy()
    for t in range(4):
        for j in range(spec.top_k):
            expect[t] += w[t, j] * indep.dense_ffn(layer, int(idx[t, j]), xf[t:t + 1])[0]
    np.testing.assert_allclose(r["out64"], expect, rtol=1e-11, atol=1e-11)
    assert np.array_equal(r["out16"], expect.astype(np.float16).view(np.uint16)) or \
        np.max(np.abs(indep.f16(r["out16"]) - expect.astype(np.float16))) <= 2.0 ** -10


def test_sampled_tokens_match_full(oracle_lib):
    spec = synth.CONFIGS["tiny"]
    layer = synth.make_layer(spec)
    x = synth.make_tokens(spec, 12)
    full = oracle_lib.forward(layer, x)
    sel = np.array([11, 0, 5])
    part = oracle_lib.forward(layer, x, tokens=sel)
    assert np.array_equal(part["out64"], full["out64"][sel])
    assert np.array_equal(part["idx"], full["idx"])


# ------------------------------------------------------------ invariants

@pytest.mark.parametrize("name", ["tiny", "e256_top8_shared", "e512_top4_shared"])
def test_routing_invariants(oracle_lib, name):
    spec = synth.CONFIGS[name]
    layer = synth.make_layer(spec, experts=False)
    n = 37
    x = synth.make_tokens(spec, n)
    k, E = spec.top_k, spec.n_experts
    r = dict(logits=oracle_lib.router_logits(x, layer.router_w, layer.router_bias))
    r["idx"], r["w"], _ = oracle_lib.topk(r["logits"], k)
    r["counts"], r["offsets"], r["perm"] = oracle_lib.group(r["idx"], E)
    np.testing.assert_allclose(r["w"].astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert r["counts"].sum() == n * k and r["offsets"][-1] == n * k
    assert np.all(np.diff(r["offsets"]) == r["counts"])
    perm = r["perm"]
    assert np.array_equal(np.sort(perm), np.arange(n * k))
    tok = perm // k
    assert np.array_equal(np.bincount(tok, minlength=n), np.full(n, k))
    for e in range(E):
        seg = perm[r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(r["idx"].reshape(-1)[seg] == e)
        assert len(np.unique(seg // k)) == len(seg)      # a token at most once per expert
        assert np.all(np.diff(seg) > 0)                  # stable


def test_zipf_bias_skews_traffic(oracle_lib):
    spec = synth.CONFIGS["e64_top2_sweep_zipf"].with_(hidden=512, inter=128)
    layer = synth.make_layer(spec, experts=False)
    x = synth.make_tokens(spec, 256)
    idx, _, _ = oracle_lib.topk(oracle_lib.router_logits(x, layer.router_w, layer.router_bias), 2)
    c, _, _ = oracle_lib.group(idx, spec.n_experts)
    assert c[:4].sum() > c[-16:].sum()


# ------------------------------------------------------------------ RMSNorm

def _h(v):
    return np.asarray(v, np.float16).view(np.uint16)


@pytest.mark.parametrize("c", [1.0, 3.0, -0.5, 100.0])
def test_rmsnorm_constant_row_is_unit(oracle_lib, c):
    """A constant row c with unit gain and eps 0 normalises to sign(c)."""
    H = 512
    xn = oracle_lib.rmsnorm(_h(np.full((2, H), c)), _h(np.ones(H)), 0.0)
    assert np.array_equal(xn, _h(np.full((2, H), math.copysign(1.0, c))))


@pytest.mark.parametrize("H", [256, 1024, 4096])
def test_rmsnorm_single_spike_is_sqrt_h(oracle_lib, H):
    """One non-zero entry a (a power of two) in a row of H (a power of 4):
    mean square a^2 / H, so the entry becomes sign(a) sqrt(H) exactly and the
    rest stay 0."""
    for j, a in [(0, 4.0), (H - 1, -0.25), (H // 2 + 3, 64.0)]:
        r = np.zeros((1, H))
        r[0, j] = a
        xn = oracle_lib.rmsnorm(_h(r), _h(np.ones(H)), 0.0).view(np.float16).astype(np.float64)
        expect = np.zeros((1, H))
        expect[0, j] = math.copysign(math.sqrt(H), a)
        assert np.array_equal(xn, expect)


def test_rmsnorm_scale_invariance_and_gain(oracle_lib):
    """Scaling a row up by a power of two (exact in fp16) leaves the output
    unchanged (eps 0), and doubling the gain doubles it, bit for bit."""
    rng = np.random.default_rng(7)
    H = 2048
    r = rng.normal(0, 1, (3, H)).astype(np.float16)
    g = rng.uniform(0.5, 1.5, H).astype(np.float16)
    base = oracle_lib.rmsnorm(r.view(np.uint16), g.view(np.uint16), 0.0)
    for k in (1, 3):
        scaled = (r.astype(np.float64) * 2.0 ** k).astype(np.float16)
        assert np.array_equal(scaled.astype(np.float64), r.astype(np.float64) * 2.0 ** k)
        assert np.array_equal(oracle_lib.rmsnorm(scaled.view(np.uint16), g.view(np.uint16), 0.0),
                              base)
    g2 = (g.astype(np.float64) * 2).astype(np.float16)
    doubled = oracle_lib.rmsnorm(r.view(np.uint16), g2.view(np.uint16), 0.0)
    assert np.array_equal(doubled.view(np.float16).astype(np.float64),
                          base.view(np.float16).astype(np.float64) * 2)


@pytest.mark.parametrize("c,eps,expect", [(1.0, 3.0, 0.5), (3.0, 7.0, 0.75), (-2.0, 12.0, -0.5),
                                          (0.5, 0.75, 0.5)])
def test_rmsnorm_eps_closed_form(oracle_lib, c, eps, expect):
    """A constant row c: mean square c^2, so the output is c / sqrt(c^2 + eps)
    times the gain; the cases are chosen so that this is a dyadic number."""
    H = 384
    g = np.linspace(0.5, 1.5, H).astype(np.float16)
    xn = oracle_lib.rmsnorm(_h(np.full((1, H), c)), g.view(np.uint16), eps)
    want = (g.astype(np.float64) * expect).astype(np.float16)
    assert np.array_equal(xn.view(np.float16), want[None, :])


def _fp16_round_decimal(v):
    """Nearest fp16 (ties to even) of a Decimal, by comparing with the two
    fp16 neighbours of a first guess in Decimal arithmetic; also returns how
    close v is to the midpoint of those neighbours (relative), so that
    near-ties can be set aside."""
    from decimal import Decimal
    g = np.float16(float(v))
    lo = np.nextafter(g, np.float16(-np.inf))
    hi = np.nextafter(g, np.float16(np.inf))
    cands = [lo, g, hi]
    dist = [abs(Decimal(float(c)) - v) for c in cands]
    best = min(range(3), key=lambda i: (dist[i], int(np.array(cands[i]).view(np.uint16)) & 1))
    srt = sorted(dist)
    gap = (srt[1] - srt[0]) / max(abs(v), Decimal("1e-30"))
    return cands[best], gap


@pytest.mark.parametrize("eps", [0.0, 1e-6, 1e-2, 4.0])
def test_rmsnorm_correctly_rounded(oracle_lib, eps):
    """Against r_h g_h / sqrt(mean(r^2) + eps) evaluated in 50-digit decimal
    arithmetic: every output is that value correctly rounded to fp16 (entries
    within 1e-12 relative of a rounding midpoint, where fp64 may decide either
    way, are set aside; there are next to none)."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    rng = np.random.default_rng(11)
    H = 1024
    r = (rng.normal(0, 1, (16, H)) * rng.choice([0.01, 1.0, 30.0], (16, 1))).astype(np.float16)
    g = rng.uniform(0.2, 2.0, H).astype(np.float16)
    got = oracle_lib.rmsnorm(r.view(np.uint16), g.view(np.uint16), eps).view(np.float16)
    e = Decimal(float(np.float32(eps)))
    skipped = 0
    for t in range(r.shape[0]):
        rd = [Decimal(float(v)) for v in r[t]]
        ms = sum((v * v for v in rd), Decimal(0)) / H
        rs = 1 / (ms + e).sqrt()
        for h in range(H):
            want, gap = _fp16_round_decimal(rd[h] * rs * Decimal(float(g[h])))
            if gap < Decimal("1e-12"):
                skipped += 1
                continue
            assert got[t, h].view(np.uint16) == np.array(want).view(np.uint16), (t, h)
    assert skipped <= 2
