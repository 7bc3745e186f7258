"""The oracle's pins catch planted mistakes.

Each case compiles a copy of the oracle source with one plausible mistake
(a flipped sign, a dropped term, a wrong tie order, a transposed operand)
and checks that at least one pin from ``test_oracle_pins`` fails on it.
The mistakes are planted in the CPU oracle only.
"""

import os

import pytest

import tests.test_oracle_pins as P
import tests.test_oracle_tree as PT

MUTATIONS = {
    "residual sign flipped": ("std::max(0.0, p[y] - q[y])", "std::max(0.0, q[y] - p[y])"),
    "accept ratio transposed": ("std::min(1.0, px / qx)", "std::min(1.0, qx / px)"),
    "saguaro factor on the wrong set": ("for (int y : S) qp[y] = C * q[y];",
                                        "for (int y : S) qp[y] = q[y] / C;"),
    "saguaro not renormalised": ("for (auto& v : qp) v /= total;", ""),
    "top-F ties to the higher index": ("(z[a] == z[b] && a < b)", "(z[a] == z[b] && a > b)"),
    "inverse CDF not strict": ("if (cum > thr) {", "if (cum >= thr) {"),
    "temperature dropped": ("std::exp((z[y] - m) / T)", "std::exp(z[y] - m)"),
    "philox key bump dropped": ("k[1] += PhiloxConst<W>::W1;", ""),
    "philox words swapped": ("c[1] = lo1;", "c[1] = lo0;"),
    "fanout exponent": ("(double)k / (1.0 + r)", "(double)k / r"),
    "per-position C collapsed to the first": ("auto qp = saguaro(q[i], S, C[i]);",
                                              "auto qp = saguaro(q[i], S, C[0]);"),
    "per-sequence temperature ignored": ("const double Tb = T_rows ? T_rows[b] : T;",
                                         "const double Tb = T;"),
    "greedy bonus from the runner-up": ("bonus[b] = top_n(zk, 1)[0];",
                                        "bonus[b] = top_n(zk, 2)[1];"),
    "tree residual not renormalised": ("for (auto& e : w) e /= Z;", ""),
    "tree accept uniform of the wrong node": ("(uint32_t)(v - 1), 0u, round)",
                                              "(uint32_t)v, 0u, round)"),
    "tree draft from the child's own row": ("((int64_t)b * N + parent[v]) * d_stride",
                                            "((int64_t)b * N + v) * d_stride"),
    "tree bonus before the last child": ("for (int v = u + 1; v < N && !moved; ++v) {",
                                         "for (int v = u + 1; v < N - 1 && !moved; ++v) {"),
}

PINS = [
    P.test_philox_round_structure_matches_numpy_philox4x64,
    P.test_softmax_matches_scipy_and_temperature,
    P.test_top_n_matches_stable_library_sort,
    lambda orc: [P.test_saguaro_closed_forms(orc, C) for C in (0.5, 0.3)],
    P.test_accept_prob_rule,
    P.test_residual_mass_is_total_variation,
    P.test_inverse_cdf_matches_library_search,
    lambda orc: P.test_losslessness_exact_enumeration(orc, 5, 3, 0.5, 1.0),
    P.test_fanout_is_the_lagrange_optimum,
    lambda orc: P.test_accept_length_law_per_position_C(orc, (0.3, 0.5, 0.8, 1.0)),
    P.test_greedy_is_the_low_temperature_limit,
    P.test_per_sequence_temperature_equals_separate_calls,
    PT.test_chain_tree_is_linear_verification,
    lambda orc: PT.test_tree_walk_laws_monte_carlo(orc, "two-by-two"),
    PT.test_tree_draft_follows_parent_distribution,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_detect_planted_mistake(orc, tmp_path, name):
    old, new = MUTATIONS[name]
    src = orc.source_text()
    assert src.count(old) == 1, name
    path = orc.build_variant(src.replace(old, new), os.path.join(str(tmp_path), "mut.so"))
    failed = []
    with orc.use_library(path):
        for pin in PINS:
            try:
                pin(orc)
            except AssertionError:
                failed.append(getattr(pin, "__name__", "lambda"))
    assert failed, f"no pin caught: {name}"
