"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

The mistake is planted in a temporary copy of the oracle's C source, compiled on
the CPU; the committed oracle is never modified.
"""
import os
import shutil
import subprocess

import pytest

import pins
from oracle import Oracle
from oracle.oracle import SRC

# (name, original text, planted text) -- each original must occur exactly once
MUTANTS = [
    ("gate_up_swapped", "h[c] = silu(g[c]) * g[I + c];", "h[c] = silu(g[I + c]) * g[c];"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("gate_up_expand_dropped", "for (int32_t n = 0; n < 2 * I; ++n) g[n] += u[n];",
     "for (int32_t n = 0; n < 2 * I; ++n) g[n] += 0.0 * u[n];"),
    ("down_expand_dropped", "for (int32_t n = 0; n < H; ++n) d[n] += u[n];",
     "for (int32_t n = 0; n < H; ++n) d[n] += 0.0 * u[n];"),
    ("expand_adapter_stride_wrong", "vecmat_bf16(B_dn + ae * r_max * H, r, H, H, s, u);",
     "vecmat_bf16(B_dn + ae * r * H, r, H, H, s, u);"),
    ("expand_transposed", "vecmat_bf16(B_gu + ae * r_max * 2 * I, r, 2 * (int64_t)I, 2 * (int64_t)I, s, u);",
     "matvec_bf16(B_gu + ae * r_max * 2 * I, 2 * (int64_t)I, r, r_max, s, u);"),
    ("shrink_reads_x_in_down", "matvec_bf16(A_dn + ae * r_max * I, r, I, I, h, s);",
     "matvec_bf16(A_dn + ae * r_max * I, r, I, I, xt, s);"),
    ("combine_weight_ignored", "o[c] += w * d[c];", "o[c] += d[c];"),
    ("no_renormalise", "for (int32_t j = 0; j < k; ++j) topk_w[t * k + j] /= chosen_sum;", ""),
    ("ties_to_higher_index", "(p[e] == p[best] && l[e] > l[best])", "(p[e] == p[best] && l[e] >= l[best])"),
    ("sort_adapter_before_expert", "if (u->e != v->e) return u->e < v->e ? -1 : 1;",
     "if (u->a != v->a) return u->a < v->a ? -1 : 1;"),
    ("no_padding", "int64_t padded = (n + BM - 1) / BM * BM;", "int64_t padded = n;"),
    ("runs_include_no_adapter", "if (a >= 0) {\n                if (nr >= cap_runs)",
     "if (a >= -1) {\n                if (nr >= cap_runs)"),
    ("invalid_adapter_kept", "if (e < 0 || e >= E || a < -1 || a >= L) { ++dropped; continue; }\n        keys",
     "if (e < 0 || e >= E) { ++dropped; continue; }\n        keys"),
    ("rank_ignored", "const int32_t r = ranks[a];\n                    const int64_t ae = (int64_t)a * E + e;\n                    /* gate_up shrink",
     "const int32_t r = r_max;\n                    const int64_t ae = (int64_t)a * E + e;\n                    /* gate_up shrink"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, planted):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} not unique"
    mut_src = tmp_path / f"oracle_{name}.c"
    mut_src.write_text(src.replace(orig, planted))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mut_src), "-o", str(lib), "-lm"],
                   check=True)
    mutant = Oracle(str(lib))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, RuntimeError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake '{name}' passed every pin"
