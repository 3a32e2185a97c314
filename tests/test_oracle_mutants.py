"""Planted mistakes: each mutant of the oracle's C source must fail a pin.

Every mutant is a plausible slip in writing the method down (a flipped sign,
a dropped log-weight, a missing max shift, eps multiplied instead of divided,
a wrong cost, a plan with g of the wrong sign).  The mutant is compiled from an
edited copy of ``oracle/sinkhorn_oracle.c`` on the CPU and swapped in for the
real oracle while the pins of ``test_oracle.py`` run; at least one pin must
fail for every mutant.
"""
import os

import pytest

import oracle as orc
from tests import test_oracle as pins

# (name, function whose body is edited, original text, mutated text)
MUTANTS = [
    ("f_logb_sign", "orc_f_update", "/ eps + lb[j];", "/ eps - lb[j];"),
    ("f_logb_dropped", "orc_f_update", "/ eps + lb[j];", "/ eps;"),
    ("f_eps_times", "orc_f_update", "(g[j] - C[i * m + j]) / eps", "(g[j] - C[i * m + j]) * eps"),
    ("f_g_sign", "orc_f_update", "(g[j] - C[i * m + j])", "(-g[j] - C[i * m + j])"),
    ("g_loga_dropped", "orc_g_update", "la[i] = log((double)a[i]);", "la[i] = 0.0;"),
    ("g_cost_sign", "orc_g_update", "(f[i] - C[i * m + j])", "(f[i] + C[i * m + j])"),
    ("lse_no_shift", "lse", "return M + log(s);", "return log(s);"),
    ("cost_abs", "sqdist", "s += t * t;", "s += fabs(t);"),
    ("plan_g_sign", "orc_apply_plan", "exp((f[i] + g[j] - C[i * m + j]) / eps)",
     "exp((f[i] - g[j] - C[i * m + j]) / eps)"),
    ("plan_no_a", "orc_apply_plan", "double p = (double)a[i] * (double)b[j]",
     "double p = (double)b[j]"),
    ("prop1_no_ynorm", "orc_f_update_prop1", "double ghat = g[j] - yy;", "double ghat = g[j];"),
    ("cosine_no_factor2", "orc_cost_cosine", "- 2.0 * cosv;", "- cosv;"),
    ("cosine_no_ynorm", "orc_cost_cosine", "dot / (nx * ny[j])", "dot / nx"),
    ("tc_no_a", "orc_transport_cost", "(double)a[i] * (double)b[j] * exp", "(double)b[j] * exp"),
    ("tc_g_sign", "orc_transport_cost", "exp((f[i] + g[j] - C[i * m + j]) / eps)",
     "exp((f[i] - g[j] - C[i * m + j]) / eps)"),
    ("marg_col_no_b", "orc_marginals", "col[j] = s;", "col[j] = s / (double)b[j];"),
]

PINS = [
    lambda: pins.test_single_pair_closed_form(),
    lambda: pins.test_one_column_closed_form(),
    lambda: pins.test_one_row_closed_form_g_update(),
    lambda: pins.test_two_points_softmin_limit(),
    lambda: pins.test_symmetric_two_by_two_converged_plan(),
    lambda: pins.test_cost_matches_scipy_cdist(),
    lambda: pins.test_proposition1_identity(17, 29, 2, 0.05),
    lambda: pins.test_marginals_exact_after_each_half(),
    lambda: pins.test_gauge_invariance_of_plan_and_update_equivariance(),
    lambda: pins.test_large_eps_plan_is_product_measure(),
    lambda: pins.test_grad_x_matches_finite_differences(),
    lambda: pins.test_cosine_cost_special_values(),
    lambda: pins.test_cosine_cost_equals_squared_euclidean_on_unit_rows(),
    lambda: pins.test_entropic_duality_links_dual_value_transport_cost_and_marginals(),
]


def _function_span(src: str, fname: str):
    start = src.index(fname + "(")
    # walk back to the start of the line holding the definition
    start = src.rfind("\n", 0, start) + 1
    depth, i = 0, src.index("{", start)
    while True:
        if src[i] == "{":
            depth += 1
        elif src[i] == "}":
            depth -= 1
            if depth == 0:
                return start, i + 1
        i += 1


@pytest.mark.parametrize("name,fname,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistakes(tmp_path, name, fname, old, new):
    src = orc.source_text()
    # the definition of fname (skip forward declarations and calls)
    key = {"lse": "static double lse(", "sqdist": "static double sqdist(",
           "orc_transport_cost": "double orc_transport_cost("}.get(fname, "void " + fname + "(")
    s0 = src.index(key)
    _, s1 = _function_span(src, key[:-1])
    body = src[s0:s1]
    assert old in body, f"mutation site for {name} not found"
    mutated = src[:s0] + body.replace(old, new) + src[s1:]
    lib = orc.compile_variant(mutated, os.path.join(str(tmp_path), f"mut_{name}.so"))
    failures = 0
    with orc.use_library(lib):
        for pin in PINS:
            try:
                pin()
            except Exception:
                failures += 1
    assert failures >= 1, f"mutant {name} passed every pin"
