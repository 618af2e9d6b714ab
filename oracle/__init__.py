"""CPU oracle for the quantised MoE layer forward.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path.  It shares no code
with the CUDA path.  Parity of every function is pinned by tests that do not
call it (brute force, exact rational arithmetic, closed forms and hand-worked
cases under ``tests/``).
"""
from .oracle import (  # noqa: F401
    build, load, OracleLayer, half_to_double, double_to_half, unpack_codes, dequant,
    router_logits, topk, group, expert_ffn, forward, rmsnorm, num_threads, set_num_threads,
)
