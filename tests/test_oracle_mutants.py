"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins in test_oracle_pins.py catch every one of them."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "gate_up_swapped": ("g / (1.0 + exp(-g)) * u", "u / (1.0 + exp(-u)) * g"),
    "zero_sign": ("(double)code_at(crow, k, wbits) - (double)zrow[g]",
                  "(double)code_at(crow, k, wbits) + (double)zrow[g]"),
    "nibble_order": ("(k & 1) ? (b >> 4) : (b & 0xF)", "(k & 1) ? (b & 0xF) : (b >> 4)"),
    "residual_dropped": ("double v = oracle_half_to_double(x[(int64_t)sel[i] * H + c]);",
                         "double v = 0.0;"),
    "topk_tie_to_higher_id": ("l[e] > l[best]", "l[e] >= l[best]"),
    "round_ties_to_odd": ("(d == bd && (bits & 1u) == 0)", "(d == bd && (bits & 1u) == 1)"),
    "round_first_guess_kept": ("for (int i = 1; i < 3; i++) {", "for (int i = 3; i < 3; i++) {"),
    "bias_dropped": ("volatile float lb = l + bias[e];", "volatile float lb = l;"),
    "shared_gate_sign": ("wt[i] = 1.0 / (1.0 + exp(-z));", "wt[i] = 1.0 / (1.0 + exp(z));"),
    "group_index": ("int g = k / group;", "int g = k % group;"),
    "slot_weight_swapped": ("v += w[(int64_t)sel[i] * k + j] * yslot",
                            "v += w[(int64_t)sel[i] * k + (k - 1 - j)] * yslot"),
    "unstable_group": ("perm[next[idx[p]]++] = (int32_t)p;",
                       "perm[offsets[idx[p] + 1] - 1 - (next[idx[p]]++ - offsets[idx[p]])]"
                       " = (int32_t)p;"),
    "down_index_transposed": ("dequant_row(codes[2] + r * rb_d", "dequant_row(codes[2] + ((r * 7) % H) * rb_d"),
    "half_rounding_truncates": ("double r = nearbyint(ldexp(m, 11));", "double r = floor(ldexp(m, 11));"),
    "rmsnorm_eps_dropped": ("sqrt(sq / H + (double)eps)", "sqrt(sq / H)"),
    "rmsnorm_mean_over_groups": ("sqrt(sq / H + (double)eps)", "sqrt(sq / (H / 128) + (double)eps)"),
    "rmsnorm_gain_dropped": ("oracle_half_to_double(row[h]) * rs * oracle_half_to_double(g[h]));",
                             "oracle_half_to_double(row[h]) * rs);"),
    "rmsnorm_square_dropped": ("sq += v * v;", "sq += fabs(v);"),
    # precision mistakes: the sum of squares or the scaled row kept in fp32
    "rmsnorm_sum_in_fp32": ("        double sq = 0.0;", "        float sq = 0.0f;"),
    "rmsnorm_rs_in_fp32": ("const double rs = 1.0 / sqrt(sq / H + (double)eps);",
                           "const double rs = (float)(1.0 / sqrt(sq / H + (double)eps));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation site not found: %s" % name
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(old, new))
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.h"), tmp_path / "oracle.h")
    so = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fopenmp", "-fPIC",
                    "-shared", "-w", "-o", str(so), str(src), "-lm"], check=True)
    env = dict(os.environ, QEFFN_ORACLE_SO=str(so), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "planted mistake %r not caught:\n%s" % (name, r.stdout[-2000:])
