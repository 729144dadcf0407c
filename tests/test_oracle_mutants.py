"""Planted mistakes in the oracle must fail its pins.

Each mutant is a copy of ``oracle/grpo_oracle.c`` with one plausible mistake
(a dropped term, a wrong sign or index, a transposed operand, the traps the
page "Making Dr GRPO go brrr" warns about), compiled on the CPU into a
temporary library.  The test requires at least one pin of
``oracle_pins.ALL_CHEAP`` to reject it.  CPU only."""
import os
import types

import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    # "The completion mask"
    "mask_drops_eos_itself": ("j <= first_eos : 1", "j < first_eos : 1"),
    "mask_argmax_trap": ("int64_t first_eos = -1;", "int64_t first_eos = 0;"),
    "mask_no_eos_all_zero": ("j <= first_eos : 1)", "j <= first_eos : 0)"),
    "len_off_by_one": ("first_eos + 1 : C", "first_eos : C"),
    # advantage
    "advantage_divides_by_G_minus_1": ("mu = sum / (double)G;\n        for (int64_t g = 0; g < G; ++g)\n            A[b * G + g] = R[b * G + g] - mu;",
                                       "mu = sum / (double)(G - 1);\n        for (int64_t g = 0; g < G; ++g)\n            A[b * G + g] = R[b * G + g] - mu;"),
    # reward contrast ("The sparse-reward bottleneck")
    "contrast_counts_uniform_groups": ("if (!all_equal)\n            useful += 1;",
                                       "if (all_equal)\n            useful += 1;"),
    "contrast_skips_last_reward": ("k < G && all_equal", "k < G - 1 && all_equal"),
    "contrast_compares_to_batch_start": ("grp[k] != grp[0]", "grp[k] != R[0]"),
    "contrast_compares_neighbours_only_once": ("for (int64_t k = 1; k < G && all_equal; ++k)",
                                              "for (int64_t k = 1; k < 2 && k < G && all_equal; ++k)"),
    # original GRPO advantage
    "std_sample_not_population": ("sqrt(ss / (double)G)", "sqrt(ss / (double)(G - 1))"),
    "std_missing_sqrt": ("double sigma = sqrt(ss / (double)G);", "double sigma = ss / (double)G;"),
    "std_not_divided": ("(R[b * G + g] - mu) / (sigma + std_eps);", "(R[b * G + g] - mu);"),
    # per-response mean aggregation
    "seq_mean_divides_by_C": ("norm * (double)(len[i] > 0 ? len[i] : 1)", "norm * (double)C"),
    "seq_mean_loss_unweighted": ("(long double)l * ((long double)norm / (long double)denom)", "(long double)l"),
    "advantage_sign": ("R[b * G + g] - mu;", "mu - R[b * G + g];"),
    # compute_logprobs
    "shift_off_by_one": ("i * c->T + (c->P - 1 + t)", "i * c->T + (c->P + t)"),
    "lse_drops_max": ("return mx + log(s);", "return log(s);"),
    "bf16_wrong_shift": ("[v] << 16;", "[v] << 8;"),
    "target_wrong_column": ("c->ids[i * c->T + c->P + t];\n    const void",
                            "c->ids[i * c->T + c->P + t - 1];\n    const void"),
    # the loss
    "ratio_inverted": ("exp(lp - old[k])", "exp(old[k] - lp)"),
    "clip_after_multiply": ("clamp_d(r, 1.0 - eps, 1.0 + eps) * a", "clamp_d(r * a, 1.0 - eps, 1.0 + eps)"),
    "min_becomes_max": ("unclipped < clipped ? unclipped : clipped",
                        "unclipped > clipped ? unclipped : clipped"),
    "surrogate_sign": ("double l = -s + beta * k3;", "double l = s + beta * k3;"),
    "kl_dropped": ("double l = -s + beta * k3;", "double l = -s;"),
    "k3_sign": ("k3 = exp(d) - d - 1.0;", "k3 = exp(d) + d - 1.0;"),
    "norm_per_response": ("agg == 0 ? (double)N * (double)C : (double)N", "agg == 0 ? (double)N : (double)N"),
    "mask_off_by_one_in_loss": ("if (t >= len[i]) {\n                if (w)", "if (t > len[i]) {\n                if (w)"),
    # the gradient
    "grad_ignores_clip": ("unclipped <= clipped ? a * r : 0.0", "a * r"),
    "grad_kl_sign": ("dk3 = 1.0 - exp(d);", "dk3 = exp(d) - 1.0;"),
    "grad_drops_onehot": ("(v == y ? 1.0 : 0.0) - p", "-p"),
    "grad_sign": ("out[v] = gw * ((v", "out[v] = -gw * ((v"),
    "grad_row_shift": ("int64_t t = pos - (c->P - 1);", "int64_t t = pos - c->P;"),
    "grad_ignores_upstream": ("c->g * c->w[k]", "c->w[k]"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique/present"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / f"{name}.so"))
    o = oracle.Oracle(lib)
    failures = []
    for pin in pins.ALL_CHEAP:
        try:
            pin(o)
        except (AssertionError, ValueError) as e:
            failures.append(pin.__name__)
            break
    assert failures, f"mutant {name} passed every pin"


# Planted mistakes in the numpy side of the oracle (the LM-head chain rule in
# oracle/__init__.py), loaded as a module of their own over the real C library.
PY_MUTANTS = {
    "lmhead_grad_rows_unshifted": ("h = H[i, P - 1:P - 1 + L]", "h = H[i, P:P + L]"),
    "lmhead_dhidden_misplaced": ("dH[i, P - 1:P - 1 + L] = dz @ W", "dH[i, P:P + L] = dz @ W"),
    "lmhead_drops_upstream": ("g * w[i, t]) for t", "w[i, t]) for t"),
    "lmhead_dweight_sign": ("dW += dzs.T @ h", "dW -= dzs.T @ h"),
    "lmhead_dweight_next_row": ("dW += dzs.T @ h", "dW += dzs.T @ H[i, P:P + L]"),
    "lmhead_dhidden_uses_transpose": ("dH[i, P - 1:P - 1 + L] = dz @ W\n",
                                      "dH[i, P - 1:P - 1 + L] = (W.T @ dz.T).T[:, ::-1]\n"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_mutant_is_caught(name):
    with open(oracle.__file__) as f:
        src = f.read()
    old, new = PY_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = oracle.__file__
    exec(compile(src.replace(old, new), oracle.__file__, "exec"), mod.__dict__)
    o = mod.Oracle(oracle.build())
    failures = []
    for pin in pins.ALL_CHEAP:
        try:
            pin(o)
        except (AssertionError, ValueError) as e:
            failures.append(pin.__name__)
            break
    assert failures, f"mutant {name} passed every pin"
