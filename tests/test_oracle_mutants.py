"""The pins are strong enough: each plausible mistake planted in a copy of the oracle
(on the CPU) must make at least one pin fail. The real oracle is never modified: C
mistakes go into a recompiled copy of its source, Python mistakes into a re-defined copy
of one method bound to a single oracle instance."""
import inspect
import textwrap
import types

import pytest

import pins
from oracle import oracle as O

# (name, text in the oracle source, replacement). Each text occurs exactly once, and every
# mutant keeps all array accesses in bounds.
MUTANTS = [
    ("sigmoid_sign", "exp(-(double)l[e])", "exp((double)l[e])"),
    ("bias_dropped", "c[e] = s[e] + bias[e];", "c[e] = s[e];"),
    ("group_score_max_only", "scratch[0].key + scratch[1].key : scratch[0].key", "scratch[0].key : scratch[0].key"),
    ("dropped_groups_scored_zero", "if (kept[e / S]) { scratch[n_cand].key = c[e];",
     "{ scratch[n_cand].key = kept[e / S] ? c[e] : 0.0f;"),
    ("ties_to_higher_index", "return (a->id > b->id) - (a->id < b->id);", "return (a->id < b->id) - (a->id > b->id);"),
    ("ascending_rank", "if (a->key > b->key) return -1;", "if (a->key < b->key) return -1;"),
    ("weights_from_biased_score", "double wk = cf->scale * (double)s[idx[k]] / sum;",
     "double wk = cf->scale * (double)c[idx[k]] / sum;"),
    ("scale_missing", "double wk = cf->scale * (double)s[idx[k]] / sum;", "double wk = (double)s[idx[k]] / sum;"),
    ("one_group_short", "for (int r = 0; r < cf->topk_group; r++) {", "for (int r = 0; r + 1 < cf->topk_group; r++) {"),
    ("gate_transposed", "x[j] * bf16_value(wg[(int64_t)i * d + j]);", "x[j] * bf16_value(wg[(int64_t)j * I + i]);"),
    ("down_transposed", "h[i] * bf16_value(wd[(int64_t)j * I + i]);", "h[i] * bf16_value(wd[(int64_t)i * d + j]);"),
    ("sigmoid_not_silu", "h[i] = g / (1.0 + exp(-g)) * u;", "h[i] = 1.0 / (1.0 + exp(-g)) * u;"),
    ("silu_on_up", "h[i] = g / (1.0 + exp(-g)) * u;", "h[i] = u / (1.0 + exp(-u)) * g;"),
    ("combine_drops_slot", "for (int k = 0; k < K; k++) acc += w64", "for (int k = 0; k + 1 < K; k++) acc += w64"),
    ("logits_transposed", "(double)wr[(int64_t)e * c->d + j]", "(double)wr[(int64_t)j * c->E + e]"),
    ("logits_kept_fp64_sigmoid_in_fp32", "s[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));",
     "s[e] = 1.0f / (1.0f + (float)exp(-(double)l[e]) * 1.0000005f);"),
    ("residual_weights_swapped", "const double a = sqrt((double)(k - 1) / (double)k), b = 1.0 / sqrt((double)k);",
     "const double b = sqrt((double)(k - 1) / (double)k), a = 1.0 / sqrt((double)k);"),
    ("residual_step_off_by_one", "const double a = sqrt((double)(k - 1) / (double)k), b = 1.0 / sqrt((double)k);",
     "const double a = sqrt((double)(k - 2) / (double)(k - 1)), b = 1.0 / sqrt((double)(k - 1));"),
    ("rmsnorm_sum_not_mean", "1.0 / sqrt(ss / (double)d + eps)", "1.0 / sqrt(ss + eps)"),
    ("rmsnorm_eps_dropped", "1.0 / sqrt(ss / (double)d + eps)", "1.0 / sqrt(ss / (double)d)"),
    ("rmsnorm_gain_dropped", "y[j] = bf16_value(gamma[j]) * v[j] * r;", "y[j] = v[j] * r;"),
    ("bf16_truncates", "double r = nearbyint(ldexp(m, 8));", "double r = trunc(ldexp(m, 8));"),
    ("e4m3_bias_off_by_one", "else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_subnormal_scale", "if (e == 0) v = ldexp((double)m / 8.0, -6);", "if (e == 0) v = ldexp((double)m / 8.0, -7);"),
    ("fp8_down_scale_dropped", "acc += h[i] * ((double)ds[j] * e4m3_value(wd_q[(int64_t)j * I + i]));",
     "acc += h[i] * e4m3_value(wd_q[(int64_t)j * I + i]);"),
    ("fp8_silu_on_up", "e4m3_value(wu_q[(int64_t)i * d + j]));\n        }\n        h[i] = g * u / (1.0 + exp(-g));",
     "e4m3_value(wu_q[(int64_t)i * d + j]));\n        }\n        h[i] = g * u / (1.0 + exp(-u));"),
    ("nvfp4_silu_on_up", "nvfp4_value(uq, ub, ut, j);\n        }\n        h[i] = g * u / (1.0 + exp(-g));",
     "nvfp4_value(uq, ub, ut, j);\n        }\n        h[i] = g * u / (1.0 + exp(-u));"),
    ("e2m1_exponent_bias_off", "ldexp(1.0 + 0.5 * (double)m, e - 1)", "ldexp(1.0 + 0.5 * (double)m, e - 2)"),
    ("e2m1_subnormal_not_halved", "e == 0 ? 0.5 * (double)m :", "e == 0 ? (double)m :"),
    ("nvfp4_nibbles_swapped", "(c & 1) ? (byte >> 4) : (byte & 15)", "(c & 1) ? (byte & 15) : (byte >> 4)"),
    ("nvfp4_blocks_of_32", "e4m3_value(bs_row[c / 16])", "e4m3_value(bs_row[c / 32])"),
    ("nvfp4_tensor_scale_dropped", "return t * e4m3_value(bs_row[c / 16])", "return e4m3_value(bs_row[c / 16])"),
    ("fp8_up_scale_from_gate", "u += x[j] * ((double)us[i] * e4m3_value(wu_q[(int64_t)i * d + j]));",
     "u += x[j] * ((double)gs[i] * e4m3_value(wu_q[(int64_t)i * d + j]));"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = open(O.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur once"
    orc = O.Oracle(O.build_variant(src.replace(old, new), name))
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, RuntimeError) as exc:  # noqa: PERF203
            caught.append((check.__name__, type(exc).__name__))
            break
    assert caught, f"no pin catches the planted mistake {name}"


# Mistakes in the Python compositions of the oracle: (name, method, text, replacement).
# _forward_with is the block composition of the FP8 and NVFP4 experts.
PY_MUTANTS = [
    ("quant_weights_from_biased_score", "_forward_with", 's = dbg["s"].astype(np.float64)',
     's = dbg["c"].astype(np.float64)'),
    ("quant_given_weights_scale_missing", "_forward_with", "w64 = shape.scale * picked / picked.sum(axis=1, keepdims=True)",
     "w64 = picked / picked.sum(axis=1, keepdims=True)"),
    ("quant_combine_drops_slot", "_forward_with", "for k in range(shape.top_k):",
     "for k in range(shape.top_k - 1):"),
    ("quant_weights_not_normalised", "_forward_with", "w64 = dbg[\"w64\"]", "w64 = dbg[\"w64\"] * 1.001"),
]


@pytest.mark.parametrize("name,method,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_is_caught(name, method, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(O.Oracle, method)))
    assert src.count(old) == 1, f"mutation anchor for {name} must occur once"
    namespace = dict(vars(O))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), namespace)  # noqa: S102
    orc = O.Oracle(O.build())
    setattr(orc, method, types.MethodType(namespace[method], orc))
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, RuntimeError) as exc:  # noqa: PERF203
            caught.append((check.__name__, type(exc).__name__))
            break
    assert caught, f"no pin catches the planted mistake {name}"
