"""Plant a plausible mistake in a copy of the oracle and check that at least
one pin fails on it.  The mistakes are planted on the CPU: in a temporary build
of the C oracle, or in a copy of the Python module that composes its steps,
loaded under another name; the real oracle is untouched."""
import os
import subprocess
import types

import pytest

from oracle_pins import ALL_PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "nvfp4_oracle.c")
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")

# (name, text in the oracle source, replacement, which occurrence (0-based))
MUTANTS = [
    ("e2m1_ties_to_lower", "(d == bestd && (c & 1) == 0 && (best & 1) == 1)", "0", 0),
    ("e4m3_ties_to_lower", "(d == bestd && (c & 1) == 0 && (best & 1) == 1)", "0", 1),
    ("e2m1_sign_dropped", "int sign = signbit(v) ? 8 : 0;", "int sign = 0;", 0),
    ("e4m3_bias_off_by_one", "ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 11)", 0),
    ("scale_divisor_dropped", "float t = ga / 6.0f;", "float t = ga;", 0),
    ("scale_without_global", "float ga = g * amax;", "float ga = amax;", 0),
    ("data_without_global", "float y = x[i] * g;", "float y = x[i];", 0),
    ("nibbles_swapped", "((lo_code & 15) | ((hi_code & 15) << 4))", "((hi_code & 15) | ((lo_code & 15) << 4))", 0),
    ("gemm_weight_scale_dropped", "((double)c->ga[m] * (double)c->gw)", "((double)c->ga[m])", 0),
    ("gemm_nibble_order", "uint8_t code = (kk & 1) ? (byte >> 4) : (byte & 15);",
     "uint8_t code = (kk & 1) ? (byte & 15) : (byte >> 4);", 0),
    ("gemm_block_scale_index", "deq_int(code, c->asf[m * (K / 16) + kk / 16])", "deq_int(code, c->asf[m * (K / 16) + kk / 32])", 0),
    ("gate_up_swapped", "double gate = y1[m * 2 * I + i];\n            double up = y1[m * 2 * I + I + i];",
     "double up = y1[m * 2 * I + i];\n            double gate = y1[m * 2 * I + I + i];", 0),
    ("silu_sign", "gate / (1.0 + exp(-gate))", "gate / (1.0 + exp(gate))", 0),
    ("route_unstable", "for (int64_t f = 0; f < R; ++f) perm[cursor[ids[f]]++] = (int32_t)f;",
     "for (int64_t f = R - 1; f >= 0; --f) perm[cursor[ids[f]]++] = (int32_t)f;", 0),
    ("validate_no_reciprocal_check", "if (!isfinite(r) || !isnormal(r)) ok = 0;", "(void)r;", 0),
    ("rmsnorm_eps_outside", "sqrt(ss / (double)H + eps)", "(sqrt(ss / (double)H) + eps)", 0),
    ("router_ties_to_higher", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])", 0),
    ("router_smallest_first", "(best < 0 || l[e] > l[best])", "(best < 0 || l[e] < l[best])", 0),
    ("ue8m0_round_to_nearest", "if (ldexp(1.0, b - 127) >= a) return b;", "if (1.5 * ldexp(1.0, b - 127) >= a) return b;", 0),
    ("ue8m0_bias_126", "return ldexp(1.0, byte - 127);", "return ldexp(1.0, byte - 126);", 0),
    ("ue8m0_no_global_scale", "float y = x[i] * g;", "float y = x[i];", 1),
    ("w4a16_silu_sign", "double silu = gate / (1.0 + exp(-gate));", "double silu = gate / (1.0 + exp(gate));", 1),
    ("w4a16_sum_not_product", "bf16_nearest(silu * up)", "bf16_nearest(silu + up)", 0),
    ("router_not_renormalised", "(float)(p[ids[t * k + j]] / zk)", "(float)(p[ids[t * k + j]])", 0),
    ("gemm_ue8m0_e4m3_decode", "orc_e2m1_value(code) * orc_ue8m0_value(sfb)", "orc_e2m1_value(code) * orc_e4m3_value(sfb)", 0),
    ("gemm_ue8m0_block_index", "deq_ue8m0(code, c->asf[m * (K / 16) + kk / 16])",
     "deq_ue8m0(code, c->asf[m * (K / 16) + kk / 32])", 0),
    ("gemm_ue8m0_weight_scale_dropped", "((double)c->ga[m] * (double)c->gw)", "((double)c->ga[m])", 1),
]


def _mutate(text, old, new, which):
    pos = -1
    for _ in range(which + 1):
        pos = text.index(old, pos + 1)
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name,old,new,which", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(orc, tmp_path, name, old, new, which):
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(mutated, encoding="utf-8")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    failed = []
    with orc.use_library(str(so)):
        for pin in ALL_PINS:
            try:
                pin(orc)
            except Exception:  # an AssertionError, or a crash of the broken maths
                failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"


# Mistakes in the composition (oracle/__init__.py): which token a permuted row
# reads, which expert's scale it takes, which rows a token subset keeps.
PY_MUTANTS = [
    ("quantize_experts_token_mod_k", "q, sf = quant_rows(xf[perm // k], g[row_e]", "q, sf = quant_rows(xf[perm % k], g[row_e]", 0),
    ("quantize_experts_unpermuted_expert", "q, sf = quant_rows(xf[perm // k], g[row_e]",
     "q, sf = quant_rows(xf[perm // k], g[np.asarray(topk_ids).reshape(-1)]", 0),
    ("quantize_experts_unpermuted_token", "q, sf = quant_rows(xf[perm // k], g[row_e]",
     "q, sf = quant_rows(xf[np.arange(T * k) // k], g[row_e]", 0),
    ("forward_subset_filter_mod_k", "rows = np.nonzero(keep[perm // k])[0]", "rows = np.nonzero(keep[perm % k])[0]", 0),
    ("forward_subset_unpermuted", "rows = np.nonzero(keep[perm // k])[0]", "rows = np.nonzero(keep[np.arange(T * k) // k])[0]", 0),
    ("forward_row_token_unpermuted", "a1q, sf1 = quant_rows(xf[perm[rows] // k]", "a1q, sf1 = quant_rows(xf[rows // k]", 0),
    ("w4a16_subset_filter_mod_k", "rows = np.nonzero(keep[perm // k])[0]", "rows = np.nonzero(keep[perm % k])[0]", 1),
]


def _load_module_copy(text):
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = PY_SRC  # the copy builds and loads the same C library
    exec(compile(text, PY_SRC, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new,which", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_composition_mutant_is_caught(orc, name, old, new, which):
    with open(PY_SRC, encoding="utf-8") as f:
        src = f.read()
    mutated = _mutate(src, old, new, which)
    assert mutated != src
    mod = _load_module_copy(mutated)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"


def test_unmutated_module_copy_passes(orc):
    """The loader itself changes nothing: the unmodified copy passes every pin."""
    with open(PY_SRC, encoding="utf-8") as f:
        mod = _load_module_copy(f.read())
    for pin in ALL_PINS:
        pin(mod)
