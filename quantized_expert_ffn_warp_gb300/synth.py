"""Seeded synthetic MoE layers and token batches in the canonical packed format.

This module only draws random numbers and lays them out in the canonical
storage format; it holds none of the layer's arithmetic.  Both the CUDA path
(through ``moe_layer_create``) and the CPU oracle consume what it returns.

Canonical packed format (one expert matrix, ``rows`` x ``K``, K contiguous):

* codes  uint8  [E, rows, K*wbits/8]. 4-bit: element k sits in byte k/2, the
  low nibble holding the even element (the packed weight block layout of
  "为什么12G显存笔记本能跑MoE-16B", section 4.2).  2-bit: element k sits in
  byte k/4, bits 2*(k%4) and 2*(k%4)+1.
* scales uint16 [E, rows, K/128]: fp16 bit patterns, one per 128-group
  (INT4 group-wise quantisation with group size 128 and one scale plus one
  zero point per group: Strata article, section 2.2).
* zeros  uint8  [E, rows, K/128]: integer zero points, one byte each.

Matrices per expert: gate (I x H), up (I x H), down (H x I).

Distributions (the workloads of the five layer shapes):

* codes uniform over all code values (a uniform byte is exactly two uniform
  nibbles or four uniform 2-bit fields),
* scales ~ U(0.005, 0.02) rounded to fp16,
* zero points ~ U{6..9} (4-bit) or U{1, 2} (2-bit: the centre of [0, 3]),
* router and shared-gate weights fp16 ~ N(0, 0.05),
* activations fp16 ~ N(0, 1),
* optional Zipf routing skew as a router bias ``-s * ln(e + 1)`` (expert 0
  hottest).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GROUP = 128
MATS = ("gate", "up", "down")


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    wbits: int = 4
    group: int = GROUP
    has_shared: bool = False
    shared_inter: int = 0
    zipf_s: Optional[float] = None
    router_std: float = 0.05
    gate_std: float = 0.05
    max_tokens: int = 1024

    def mat_shape(self, m: int, shared: bool = False):
        """(rows, K) of matrix m (0 gate, 1 up, 2 down)."""
        inter = self.shared_inter if shared else self.inter
        return (inter, self.hidden) if m < 2 else (self.hidden, inter)

    def with_(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass
class PackedLayer:
    spec: LayerSpec
    codes: list          # 3 x uint8 [E, rows, K*wbits/8]
    scales: list         # 3 x uint16 [E, rows, K/128]
    zeros: list          # 3 x uint8 [E, rows, K/128]
    router_w: np.ndarray  # uint16 [E, H]
    router_bias: Optional[np.ndarray]  # float32 [E] or None
    sh_codes: Optional[list] = None    # 3 x uint8 [1, rows, ...]
    sh_scales: Optional[list] = None
    sh_zeros: Optional[list] = None
    sh_gate_w: Optional[np.ndarray] = None  # uint16 [H]

    def nbytes_expert(self) -> int:
        """Canonical bytes of one routed expert (codes + scales + zeros)."""
        return sum(int(a[0].nbytes) for a in self.codes + self.scales + self.zeros)

    def nbytes_shared(self) -> int:
        if not self.spec.has_shared:
            return 0
        return sum(int(a.nbytes) for a in self.sh_codes + self.sh_scales + self.sh_zeros)


# The five layer shapes.  Token counts per shape are listed in TOKENS.
CONFIGS = {
    "tiny": LayerSpec("tiny", hidden=256, inter=512, n_experts=8, top_k=2, max_tokens=64),
    "e64_top2_zipf": LayerSpec("e64_top2_zipf", hidden=4096, inter=4096, n_experts=64,
                               top_k=2, zipf_s=1.1, max_tokens=64),
    "e256_top8_shared": LayerSpec("e256_top8_shared", hidden=2048, inter=512, n_experts=256,
                                  top_k=8, has_shared=True, shared_inter=512, max_tokens=64),
    "e512_top4_shared": LayerSpec("e512_top4_shared", hidden=4096, inter=1024, n_experts=512,
                                  top_k=4, has_shared=True, shared_inter=1024, zipf_s=1.0,
                                  max_tokens=64),
    "e512_top4_shared_2bit": LayerSpec("e512_top4_shared_2bit", hidden=4096, inter=1024,
                                       n_experts=512, top_k=4, wbits=2, has_shared=True,
                                       shared_inter=1024, zipf_s=1.0, max_tokens=64),
    "e64_top2_sweep": LayerSpec("e64_top2_sweep", hidden=4096, inter=14336, n_experts=64,
                                top_k=2, max_tokens=1024),
    "e64_top2_sweep_zipf": LayerSpec("e64_top2_sweep_zipf", hidden=4096, inter=14336,
                                     n_experts=64, top_k=2, zipf_s=1.2, max_tokens=1024),
    # the sweep's expert shape with 16 experts (1.4 GB of weights): small
    # enough for profiler captures of the large-batch kernels
    "e16_top2_wide": LayerSpec("e16_top2_wide", hidden=4096, inter=14336, n_experts=16,
                               top_k=2, max_tokens=1024),
}

TOKENS = {
    "tiny": (4,),
    "e64_top2_zipf": (8,),
    "e256_top8_shared": (1, 16),
    "e512_top4_shared": (1, 4, 32),
    "e512_top4_shared_2bit": (1, 4, 32),
    "e64_top2_sweep": (1, 8, 64, 256, 1024),
    "e64_top2_sweep_zipf": (1, 8, 64, 256, 1024),
    "e16_top2_wide": (256,),
}

_CONFIG_IDS = {name: i + 1 for i, name in enumerate(CONFIGS)}


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def _f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype(np.float16)).view(np.uint16)


def pack_codes(q: np.ndarray, wbits: int) -> np.ndarray:
    """Pack integer codes [..., K] into the canonical byte layout."""
    q = np.asarray(q)
    if wbits == 4:
        q = q.astype(np.uint8) & 0xF
        return np.ascontiguousarray(q[..., 0::2] | (q[..., 1::2] << 4))
    if wbits == 2:
        q = q.astype(np.uint8) & 0x3
        return np.ascontiguousarray(q[..., 0::4] | (q[..., 1::4] << 2)
                                    | (q[..., 2::4] << 4) | (q[..., 3::4] << 6))
    raise ValueError("wbits must be 4 or 2")


def _matrix_set(spec: LayerSpec, rngs, n_exp: int, shared: bool):
    codes, scales, zeros = [], [], []
    zlo, zhi = (6, 9) if spec.wbits == 4 else (1, 2)
    for m in range(3):
        rows, K = spec.mat_shape(m, shared)
        rc, rs, rz = rngs[3 * m], rngs[3 * m + 1], rngs[3 * m + 2]
        nbytes = K * spec.wbits // 8
        codes.append(rc.integers(0, 256, size=(n_exp, rows, nbytes), dtype=np.uint8))
        g = K // spec.group
        scales.append(_f16_bits(rs.uniform(0.005, 0.02, size=(n_exp, rows, g))))
        zeros.append(rz.integers(zlo, zhi + 1, size=(n_exp, rows, g), dtype=np.uint8))
    return codes, scales, zeros


def zipf_bias(n_experts: int, s: float) -> np.ndarray:
    """Per-expert router bias -s*ln(e+1): expert 0 is the hottest."""
    return (-s * np.log(np.arange(1, n_experts + 1, dtype=np.float64))).astype(np.float32)


def make_layer(spec: LayerSpec, seed: int = 0, experts: bool = True) -> PackedLayer:
    """Seeded random layer of the given shape (seed 0 = the shape's own stream).
    experts=False draws only the router (and shared gate) weights."""
    _check(spec)
    base = _CONFIG_IDS.get(spec.name, 97) * 1000003 + seed
    r = _streams(base, 24)
    codes = scales = zeros = None
    if experts:
        codes, scales, zeros = _matrix_set(spec, r[0:9], spec.n_experts, False)
    router_w = _f16_bits(r[9].normal(0.0, spec.router_std, size=(spec.n_experts, spec.hidden)))
    bias = zipf_bias(spec.n_experts, spec.zipf_s) if spec.zipf_s else None
    layer = PackedLayer(spec, codes, scales, zeros, router_w, bias)
    if spec.has_shared:
        if experts:
            layer.sh_codes, layer.sh_scales, layer.sh_zeros = _matrix_set(spec, r[10:19], 1, True)
        layer.sh_gate_w = _f16_bits(r[19].normal(0.0, spec.gate_std, size=(spec.hidden,)))
    return layer


def make_tokens(spec: LayerSpec, n: int, seed: int = 0, batch: int = 0) -> np.ndarray:
    """fp16 bit patterns [n, H] of activations ~ N(0, 1)."""
    ss = np.random.SeedSequence([_CONFIG_IDS.get(spec.name, 97), 7919, seed, batch])
    return _f16_bits(np.random.default_rng(ss).normal(0.0, 1.0, size=(n, spec.hidden)))


def make_residual(spec: LayerSpec, n: int, seed: int = 0, batch: int = 0) -> np.ndarray:
    """fp16 bit patterns [n, H] of a residual stream in front of the RMSNorm:
    N(0, 1) with about one entry in 256 scaled by 20 (outlier channels of
    hidden states; the pages give no distribution)."""
    ss = np.random.SeedSequence([_CONFIG_IDS.get(spec.name, 97), 104729, seed, batch])
    rng = np.random.default_rng(ss)
    r = rng.normal(0.0, 1.0, size=(n, spec.hidden))
    r *= np.where(rng.random(size=(n, spec.hidden)) < 1.0 / 256, 20.0, 1.0)
    return _f16_bits(r)


def make_norm_gain(spec: LayerSpec, seed: int = 0) -> np.ndarray:
    """fp16 bit patterns [H] of an RMSNorm gain ~ U(0.5, 1.5)."""
    ss = np.random.SeedSequence([_CONFIG_IDS.get(spec.name, 97), 130363, seed])
    return _f16_bits(np.random.default_rng(ss).uniform(0.5, 1.5, size=spec.hidden))


def layer_from_codes(spec: LayerSpec, q, scales, zeros, router_w, router_bias=None,
                     sh_q=None, sh_scales=None, sh_zeros=None, sh_gate_w=None) -> PackedLayer:
    """Build a layer from explicit integer codes q[m] [E, rows, K], fp16 scales
    (float arrays), integer zeros and fp16 router weights (float arrays)."""
    _check(spec)
    codes = [pack_codes(q[m], spec.wbits) for m in range(3)]
    sc = [_f16_bits(np.asarray(s, dtype=np.float64)) for s in scales]
    zs = [np.ascontiguousarray(np.asarray(z, dtype=np.uint8)) for z in zeros]
    rw = _f16_bits(np.asarray(router_w, dtype=np.float64))
    rb = None if router_bias is None else np.ascontiguousarray(np.asarray(router_bias, np.float32))
    layer = PackedLayer(spec, codes, sc, zs, rw, rb)
    if spec.has_shared:
        layer.sh_codes = [pack_codes(sh_q[m], spec.wbits) for m in range(3)]
        layer.sh_scales = [_f16_bits(np.asarray(s, dtype=np.float64)) for s in sh_scales]
        layer.sh_zeros = [np.ascontiguousarray(np.asarray(z, dtype=np.uint8)) for z in sh_zeros]
        layer.sh_gate_w = _f16_bits(np.asarray(sh_gate_w, dtype=np.float64))
    return layer


def _check(spec: LayerSpec):
    if spec.wbits not in (4, 2):
        raise ValueError("wbits must be 4 or 2")
    if spec.hidden % spec.group or spec.inter % spec.group:
        raise ValueError("hidden and inter must be multiples of the group size")
    if spec.has_shared and spec.shared_inter % spec.group:
        raise ValueError("shared_inter must be a multiple of the group size")
    if not 1 <= spec.top_k <= spec.n_experts:
        raise ValueError("need 1 <= top_k <= n_experts")


def algorithmic_bytes(layer: PackedLayer, touched_experts: int, n_tokens: int) -> int:
    """Bytes a forward call must move at minimum: the touched experts' codes,
    scales and zeros, the shared expert, the router (and shared gate) weights,
    the activations read and the outputs written."""
    s = layer.spec
    b = touched_experts * layer.nbytes_expert() + layer.nbytes_shared()
    b += layer.router_w.nbytes + (layer.router_bias.nbytes if layer.router_bias is not None else 0)
    if s.has_shared:
        b += layer.sh_gate_w.nbytes
    b += 2 * n_tokens * s.hidden * 2
    return b


def algorithmic_flops(spec: LayerSpec, n_tokens: int) -> int:
    """2*3*H*I*n*k for the routed experts, the shared expert, and the router."""
    f = 2 * 3 * spec.hidden * spec.inter * n_tokens * spec.top_k
    if spec.has_shared:
        f += 2 * 3 * spec.hidden * spec.shared_inter * n_tokens
    f += 2 * spec.n_experts * spec.hidden * n_tokens
    return f


def make_layer_device(spec: LayerSpec, seed: int = 0, device="cuda") -> dict:
    """The same distributions as make_layer, drawn on the device by a seeded
    torch generator (a different random stream from make_layer's): canonical
    buffers as device tensors (fp16 bit patterns as int16), ready for
    moe_layer_create.  Used where a layer is only timed, never checked
    against the CPU oracle, so that multi-GB layers need no host-side draw
    and copy."""
    import torch
    _check(spec)
    g = torch.Generator(device=device)
    g.manual_seed(_CONFIG_IDS.get(spec.name, 97) * 1000003 + seed)
    zlo, zhi = (6, 9) if spec.wbits == 4 else (1, 2)

    def mats(n_exp, shared):
        codes, scales, zeros = [], [], []
        for m in range(3):
            rows, K = spec.mat_shape(m, shared)
            codes.append(torch.randint(0, 256, (n_exp, rows, K * spec.wbits // 8),
                                       dtype=torch.uint8, device=device, generator=g))
            gr = K // spec.group
            s = torch.empty((n_exp, rows, gr), dtype=torch.float32, device=device)
            s.uniform_(0.005, 0.02, generator=g)
            scales.append(s.half().view(torch.int16))
            zeros.append(torch.randint(zlo, zhi + 1, (n_exp, rows, gr), dtype=torch.uint8,
                                       device=device, generator=g))
        return codes, scales, zeros

    d = {}
    d["codes"], d["scales"], d["zeros"] = mats(spec.n_experts, False)
    rw = torch.empty((spec.n_experts, spec.hidden), dtype=torch.float32, device=device)
    rw.normal_(0.0, spec.router_std, generator=g)
    d["router_w"] = rw.half().view(torch.int16)
    d["router_bias"] = (torch.from_numpy(zipf_bias(spec.n_experts, spec.zipf_s)).to(device)
                        if spec.zipf_s else None)
    if spec.has_shared:
        d["sh_codes"], d["sh_scales"], d["sh_zeros"] = mats(1, True)
        gw = torch.empty(spec.hidden, dtype=torch.float32, device=device)
        gw.normal_(0.0, spec.gate_std, generator=g)
        d["sh_gate_w"] = gw.half().view(torch.int16)
    return d


def expert_bytes(spec: LayerSpec, shared: bool = False) -> int:
    """Canonical bytes of one expert: codes, fp16 scales and byte zero points
    of its three matrices."""
    inter = spec.shared_inter if shared else spec.inter
    if shared and not spec.has_shared:
        return 0
    w = 3 * spec.hidden * inter
    return w * spec.wbits // 8 + (w // spec.group) * 3


def spec_algorithmic_bytes(spec: LayerSpec, touched_experts: float, n_tokens: int) -> float:
    """algorithmic_bytes from the shape alone."""
    b = touched_experts * expert_bytes(spec) + expert_bytes(spec, True)
    b += spec.n_experts * spec.hidden * 2 + (spec.n_experts * 4 if spec.zipf_s else 0)
    if spec.has_shared:
        b += spec.hidden * 2
    b += 2 * n_tokens * spec.hidden * 2
    return b
