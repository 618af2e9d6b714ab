"""Expert residency tiers, host side (no GPU): the placement policy
moe_residency_plan (the most frequently routed experts stay resident, ties to
the lower id) against a plain sort, and argument errors of
moe_layer_set_residency returned before any CUDA call."""
import ctypes as C

import numpy as np
import pytest


@pytest.fixture(scope="module")
def moe():
    from quantized_expert_ffn_warp_gb300 import build, moe as m
    build.build()
    m.load_library()
    return m


def _expected(counts, r):
    # stable sort by descending count: equal counts keep increasing ids
    order = sorted(range(len(counts)), key=lambda e: (-counts[e], e))
    return order[:r]


@pytest.mark.parametrize("seed", range(6))
def test_plan_is_top_r_by_count(moe, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 600))
    counts = rng.integers(0, 5, E)            # many ties
    for r in sorted({0, 1, E // 3, E // 2, E}):
        got = moe.residency_plan(counts, r)
        assert list(got) == _expected(list(counts), r)


def test_plan_zipf_keeps_hot_experts(moe):
    """Counts drawn with a Zipf skew: the plan keeps the head."""
    E = 64
    w = 1.0 / np.arange(1, E + 1) ** 1.1
    counts = np.random.default_rng(3).multinomial(20000, w / w.sum())
    got = moe.residency_plan(counts, 16)
    assert set(got) == set(np.argsort(-counts, kind="stable")[:16])
    assert 0 in got and 1 in got


def test_plan_and_residency_argument_errors(moe):
    lib = moe.load_library()
    c = np.zeros(8, np.int64)
    out = np.zeros(8, np.int32)
    P = lambda a: a.ctypes.data_as(C.c_void_p)
    assert lib.moe_residency_plan(None, 8, 2, P(out)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_residency_plan(P(c), 0, 0, P(out)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_residency_plan(P(c), 8, 9, P(out)) == moe.MOE_ERR_INVALID_ARG
    c[3] = -1
    assert lib.moe_residency_plan(P(c), 8, 2, P(out)) == moe.MOE_ERR_INVALID_ARG
    assert "negative" in lib.moe_last_error().decode()
    assert lib.moe_layer_set_residency(None, P(out), 2, 4) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_tier_stats(None, None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_ep_argument_errors_before_cuda(moe):
    """moe_ep_dispatch / moe_ep_combine refuse bad arguments before any CUDA
    call (fake pointers are never dereferenced)."""
    lib = moe.load_library()
    f = C.c_void_p(256)
    assert lib.moe_ep_dispatch(None, 1, 128, f, 1, 8, 2, f, f, f, f, f, None) == -1
    assert lib.moe_ep_dispatch(f, 1, 128, f, 1, 8, 40, f, f, f, f, f, None) == -1
    assert lib.moe_ep_dispatch(f, 1, 100, f, 1, 8, 2, f, f, f, f, f, None) == -1
    assert lib.moe_ep_dispatch(f, 1, 128, f, 3, 2, 2, f, f, f, f, f, None) == -1
    assert lib.moe_ep_combine(f, 1, 128, 1, f, f, f, f, None, 1, C.c_void_p(512), None) == -1
    assert lib.moe_ep_combine(f, 1, 128, 1, f, f, f, None, None, 1, f, None) == -1
    assert "overlaps" in lib.moe_last_error().decode()
    assert lib.moe_ep_combine(f, 1, 128, 1, f, f, f, None, None, 2, C.c_void_p(4096), None) == -1
