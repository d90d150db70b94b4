"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant is a text edit of the oracle's C source compiled to a separate
library; the pin battery (hand-worked examples, dense brute force, finite
differences, plan recount) must fail for every one of them.
"""
import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_reduce_pins as reduce_pins
from tests import test_oracle_spmm_pins as spmm_pins
from tests import test_oracle_reorder_pins as reorder_pins
from tests import test_oracle_tile_pins as tile_pins

MUTANTS = {
    "drop_dot_scale": ("return scale * s;", "return s;"),
    "softmax_jacobian_sign": ("p[e * H + h] * (ds[e * H + h] - delta)",
                              "p[e * H + h] * (ds[e * H + h] + delta)"),
    "leaky_grad_no_slope": ("z > 0.0 ? 1.0 : slope;", "z > 0.0 ? 1.0 : 0.0;"),
    "leaky_grad_one_at_kink": ("z > 0.0 ? 1.0 : slope;", "z >= 0.0 ? 1.0 : slope;"),
    "gather_destination_value": ("const double* v = V + (int64_t)col[e] * HD;",
                                 "const double* v = V + node_of(row_ids, r) * HD;"),
    "lse_without_log": ("lse[r * H + h] = m + log(z);", "lse[r * H + h] = m + z;"),
    "da_without_leaky": ("da[h * D + d] += w * leaky(z, slope);", "da[h * D + d] += w * z;"),
    "dv_uses_ds": ("dv[d] += pe * g[h * D + d];", "dv[d] += w * g[h * D + d];"),
    "dk_uses_k": ("dk[d] += w * scale * q[d];", "dk[d] += w * scale * k[d];"),
    "csc_reverse_rows": ("for (int32_t i = 0; i < N; ++i)\n    for (int64_t e = ptr[i];",
                         "for (int32_t i = N - 1; i >= 0; --i)\n    for (int64_t e = ptr[i];"),
    "chunk_off_by_one": ("if (d <= T) { light[nl++] = i; continue; }",
                         "if (d < T) { light[nl++] = i; continue; }"),
    "tile_threshold_strict": ("if (t - s >= min_count) {", "if (t - s > min_count) {"),
    "tile_keeps_duplicates": ("if (pair_count[r * 128 + c] == 1) {",
                              "if (pair_count[r * 128 + c] >= 1) {"),
    "tile_mask_column_order": ("mk[r * 4 + c / 32] |= 1u << (c % 32);",
                               "mk[r * 4 + c % 4] |= 1u << (c / 4);"),
    "rcm_not_reversed": ("for (int32_t i = 0; i < N; ++i) perm[i] = order[N - 1 - i];",
                         "for (int32_t i = 0; i < N; ++i) perm[i] = order[i];"),
    "rcm_neighbours_by_id": ("if (!seen[w]) { nb[m].key = deg[w]; nb[m].id = w; ++m; }",
                             "if (!seen[w]) { nb[m].key = 0; nb[m].id = w; ++m; }"),
    "degree_order_in_only": ("deg[i] += indptr[i + 1] - indptr[i];\n      for (int64_t e = indptr[i]; e < indptr[i + 1]; ++e) deg[indices[e]] += 1;",
                             "deg[i] += indptr[i + 1] - indptr[i];"),
    "permute_keeps_old_ids": ("indices_out[o++] = inv[indices[e]];",
                              "indices_out[o++] = indices[e];"),
    "pool_tie_largest_id": ("(v == best && j < who);", "(v == best && j > who);"),
    "pool_min_as_max": ("(op == 0 ? v > best : v < best)", "(v > best)"),
    "pool_grad_to_row": ("if (j >= 0) dx[(int64_t)j * F + f] += dout[r * F + f];",
                         "if (j >= 0) dx[r * F + f] += dout[r * F + f];"),
    "spmm_drops_weight": ("for (int64_t f = 0; f < F; ++f) yr[f] += w[e] * xj[f];",
                          "for (int64_t f = 0; f < F; ++f) yr[f] += xj[f];"),
    "spmm_row_gather": ("const double* xj = x + (int64_t)col[e] * F;",
                        "const double* xj = x + r * F;"),
}


def _battery():
    """Run the pins; return the names of those that fail."""
    failed = []
    checks = [
        ("worked_dot", lambda: pins.test_worked_example("dot_worked_example.json", oracle.DOT)),
        ("worked_gatv2", lambda: pins.test_worked_example("gatv2_worked_example.json",
                                                          oracle.GATV2)),
        ("dense_dot", lambda: pins.test_dense_bruteforce(oracle.DOT, 1, 24, 2, 4)),
        ("dense_gatv2", lambda: pins.test_dense_bruteforce(oracle.GATV2, 1, 24, 2, 4)),
        ("fd_dot", lambda: pins.test_finite_differences(oracle.DOT)),
        ("fd_gatv2", lambda: pins.test_finite_differences(oracle.GATV2)),
        ("kink", lambda: pins.test_leaky_derivative_at_zero_takes_the_slope(0.2)),
        ("plan", lambda: pins.test_plan_recount(10, 200, 6.0, 8, 4)),
        ("plan_T", lambda: pins.test_plan_recount(11, 500, 20.0, 32, 16)),
        ("tile_split", lambda: tile_pins.test_tile_split_recount(0, 300, [(0, 0), (1, 2)], 0.3,
                                                                 400, 30, 1000)),
        ("tile_threshold", tile_pins.test_tile_threshold_is_inclusive),
        ("tile_dups", tile_pins.test_tile_duplicates_stay_residual),
        ("rcm_small", reorder_pins.test_rcm_path_and_star),
        ("rcm_order", lambda: reorder_pins.test_rcm_is_a_cuthill_mckee_order(2, 150, 8.0)),
        ("degree", reorder_pins.test_degree_order),
        ("permute", reorder_pins.test_permuted_csr_is_the_relabelled_graph),
        ("pool_ties", reduce_pins.test_pooling_ties_pick_the_smallest_source),
        ("pool_brute", lambda: reduce_pins.test_pooling_brute_force(oracle.MIN, 0, 50, 4.0, 8)),
        ("pool_fd", lambda: reduce_pins.test_pooling_backward_finite_differences(oracle.MAX)),
        ("spmm_hand", spmm_pins.test_spmm_hand_example),
        ("spmm_scipy", lambda: spmm_pins.test_spmm_equals_scipy(0, 300, 6.0, 16)),
    ]
    for name, fn in checks:
        try:
            fn()
        except (AssertionError, ValueError, RuntimeError):
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant):
    old, new = MUTANTS[mutant]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {mutant} not unique"
    with oracle.variant(src.replace(old, new), mutant):
        failed = _battery()
    assert failed, f"no pin caught mutant {mutant}"
