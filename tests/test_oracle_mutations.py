"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake (a dropped term, a wrong sign, a wrong index or
comparison) in a temporary copy of the oracle's C source, builds it with gcc
and runs a selection of the pins against it; at least one pin must fail.  The
committed oracle source is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle
from tests import test_oracle_hand_trees as hand
from tests import test_oracle_pins as pins
from tests import test_oracle_predict as tp
from tests import test_oracle_budget as tb
from tests import test_oracle_logistic as tl
from tests import test_oracle_update as tu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "parent score sign": ("return 0.5 * ((sL + sR) - sP) - gamma;", "return 0.5 * ((sL + sR) + sP) - gamma;"),
    "weight sign": ("return -G / (H + lambda);", "return G / (H + lambda);"),
    "lambda dropped from score": ("return (G * G) / (H + lambda);", "return (G * G) / (H);"),
    "gamma dropped": ("return 0.5 * ((sL + sR) - sP) - gamma;", "return 0.5 * ((sL + sR) - sP);"),
    "routing < instead of <=": ("if (col[rows[k]] <= b) dst[w++] = rows[k];", "if (col[rows[k]] < b) dst[w++] = rows[k];"),
    "tie-break keeps the later candidate": ("if (!out->valid || gain > out->gain) {", "if (!out->valid || gain >= out->gain) {"),
    "min_samples_leaf strict": ("if (!(cL >= msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;\n      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);\n      if (!out->valid",
                                "if (!(cL > msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;\n      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);\n      if (!out->valid"),
    "right sum uses +": ("double GR = G_P - GL, HR = H_P - HL;\n      if (!(cL >= msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;\n      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);\n      if (!out->valid",
                         "double GR = G_P + GL, HR = H_P - HL;\n      if (!(cL >= msl && cR >= msl && HL >= mcw && HR >= mcw && HL > 0.0 && HR > 0.0)) continue;\n      double gain = orc_gain(GL, HL, GR, HR, G_P, H_P, lambda, gamma);\n      if (!out->valid"),
    "last threshold skipped": ("for (int32_t b = 0; b <= nb - 2; ++b) {\n      GL += gg[b];\n      HL += hh[b];\n      cL += c[b];\n      int64_t cR = n_P - cL;\n      double GR",
                               "for (int32_t b = 0; b <= nb - 3; ++b) {\n      GL += gg[b];\n      HL += hh[b];\n      cL += c[b];\n      int64_t cR = n_P - cL;\n      double GR"),
    "prediction update sign": ("pred[rows[k]] = pred[rows[k]] + step;", "pred[rows[k]] = pred[rows[k]] - step;"),
    "quantile index off by one": ("int64_t pk = ((int64_t)k * N + B - 1) / B - 1;", "int64_t pk = ((int64_t)k * N + B - 1) / B;"),
    "initial prediction": ("const double init = logistic ? 0.0 : sum / (double)N;",
                           "const double init = logistic ? 0.0 : sum / (double)(N + 1);"),
    "gradient sign": ("g[i] = pred[i] - (double)label[i];", "g[i] = (double)label[i] - pred[i];"),
    "raw routing >= instead of >": ("v = x > thr ? tn[v].right : tn[v].left;", "v = x >= thr ? tn[v].right : tn[v].left;"),
    "raw routing children swapped": ("v = x > thr ? tn[v].right : tn[v].left;", "v = x > thr ? tn[v].left : tn[v].right;"),
    "raw prediction without learning rate": ("const double step = lr * tn[v].leaf_value;\n      pred = pred + step;",
                                             "const double step = tn[v].leaf_value;\n      pred = pred + step;"),
    "budget keeps the lowest gains": ("if (lvl_do[j] && (lvl_gain[j] > lvl_gain[i] || (lvl_gain[j] == lvl_gain[i] && j < i))) ++rank;",
                                      "if (lvl_do[j] && (lvl_gain[j] < lvl_gain[i] || (lvl_gain[j] == lvl_gain[i] && j < i))) ++rank;"),
    "budget one leaf too many": ("const int32_t K = p->num_leaves - (leaves_done + nl);", "const int32_t K = p->num_leaves + 1 - (leaves_done + nl);"),
    "sigmoid sign": ("const double p = 1.0 / (1.0 + exp(-pred[i]));", "const double p = 1.0 / (1.0 + exp(pred[i]));"),
    "logistic hessian is p": ("if (h) h[i] = p * (1.0 - p);", "if (h) h[i] = p;"),
    "histogram H ignores the hessian": ("hh[b] += h ? h[r] : 1.0;", "hh[b] += 1.0;"),
    "node H ignores the hessian": ("HP += hv ? hv[rows[k]] : 1.0;", "HP += 1.0;"),
    "level histograms ignore the hessian": ("      H[o] += hr;", "      H[o] += 1.0;"),
    "update step subtracted": ("    pred[i] = pred[i] + step;", "    pred[i] = pred[i] - step;"),
    "update without learning rate": ("const double step = lr * leaf_value[node_of_row[i]];",
                                     "const double step = leaf_value[node_of_row[i]];"),
    "update reads the leaf of the row index": ("const double step = lr * leaf_value[node_of_row[i]];",
                                               "const double step = lr * leaf_value[i];"),
    "update fused multiply-add": ("const double step = lr * leaf_value[node_of_row[i]];\n    pred[i] = pred[i] + step;",
                                  "pred[i] = fma(lr, leaf_value[node_of_row[i]], pred[i]);"),
    "feature index transposed": ("const uint8_t* col = bins + (int64_t)j * N;\n    uint32_t* c", "const uint8_t* col = bins + (int64_t)(F - 1 - j) * N;\n    uint32_t* c"),
}

PINS = [
    ("hand single split", lambda o: hand.test_hand_tree_single_split(o)),
    ("hand two trees", lambda o: hand.test_hand_tree_two_trees_lambda_one(o)),
    ("hand gamma 8", lambda o: hand.test_hand_tree_validity_rules(o, dict(gamma=8.0), None)),
    ("hand msl 2", lambda o: hand.test_hand_tree_validity_rules(o, dict(min_samples_leaf=2), (0, 1))),
    ("tie feature", lambda o: hand.test_tie_break_prefers_smaller_feature(o)),
    ("cart", lambda o: [pins.test_depth1_tree_is_cart_stump(o, s) for s in range(3)]),
    ("brute", lambda o: [pins.test_root_split_matches_brute_force(o, s) for s in range(12)]),
    ("quantize balanced", lambda o: pins.test_quantize_all_distinct_balanced(o, 1000, 32)),
    ("invariants", lambda o: pins.test_training_invariants(o, "tiny", None, 3)),
    ("predict hand", lambda o: tp.test_hand_model(o)),
    ("budget truncation", lambda o: [tb.test_budget_tree_is_the_truncated_level_wise_tree("mid", 4000, 5, 12, o=o),
                                     tb.test_budget_tree_is_the_truncated_level_wise_tree("covtype", 6000, 6, 40, o=o)]),
    ("logistic gradients", lambda o: tl.test_gradients_closed_form(o)),
    ("logistic hand tree", lambda o: tl.test_hand_tree_depth_one(o)),
    ("logistic second tree", lambda o: tl.test_second_tree_uses_new_margins(o)),
    ("logistic histograms", lambda o: tl.test_histograms_with_hessians_brute_force(o)),
    ("update hand values", lambda o: tu.test_hand_values_exact_fractions(o)),
    ("update rounding order", lambda o: tu.test_product_rounded_before_the_sum(o)),
    ("predict = training",
     lambda o: tp.test_prediction_of_training_rows_equals_training_predictions("tiny", 3, 2, o=o)),
]


def _run_pins_against(src: str, so: str) -> list:
    """Run the pins against a mutant build; returns the names of the pins that failed."""
    oracle._SRC, oracle._LIB, oracle._lib = src, so, None
    caught = []
    for pin_name, pin in PINS:
        try:
            pin(oracle)
        except (AssertionError, oracle.OracleError):
            caught.append(pin_name)
    return caught


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/missing: {name}"
    mut_src = tmp_path / "gbdt_oracle_mut.c"
    mut_src.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so), str(mut_src),
                    "-lm"], check=True, capture_output=True)
    # a separate process, so that a mutant that reads out of bounds cannot take the suite down
    r = subprocess.run([sys.executable, "-c",
                        "import sys; from tests.test_oracle_mutations import _run_pins_against as r; "
                        "c = r(sys.argv[1], sys.argv[2]); print(c); sys.exit(1 if c else 0)",
                        str(mut_src), str(so)], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake '{name}'"


def test_control_unmutated_oracle_passes_runner(tmp_path):
    # Guards the test above: the same runner on the unmodified source must report no failure.
    mut_src = tmp_path / "gbdt_oracle_copy.c"
    mut_src.write_text(open(oracle._SRC).read())
    so = tmp_path / "libcopy.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so), str(mut_src),
                    "-lm"], check=True, capture_output=True)
    r = subprocess.run([sys.executable, "-c",
                        "import sys; from tests.test_oracle_mutations import _run_pins_against as r; "
                        "c = r(sys.argv[1], sys.argv[2]); print(c); sys.exit(1 if c else 0)",
                        str(mut_src), str(so)], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
