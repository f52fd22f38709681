"""Plant a mistake in a copy of the oracle (CPU only) and check that the pins
catch it.

Each mutant is one plausible error in restating the pages' definitions: a
dropped or reordered term, FMA contraction, the wrong tie rule, a non-strict
radius test, the radius squared in double, a wrong start, padding or returned
distance.  The copy is compiled to a temporary library and swapped in; the
real oracle is restored afterwards.  The pins are the functions of
test_oracle_pins.py, called directly.
"""
import os

import pytest

import test_oracle_ext_pins as ext
import test_oracle_knn_d_pins as kd
import test_oracle_pins as pins

# (name, text to replace in pc_oracle.c, replacement)
MUTANTS = [
    ("dropped_z_term", "return sxy + zz;", "return sxy;"),
    ("reordered_sum", "float sxy = xx + yy;\n    return sxy + zz;",
     "float syz = yy + zz;\n    return xx + syz;"),
    ("fma_contraction", "float sxy = xx + yy;\n    return sxy + zz;",
     "return fmaf(dz, dz, fmaf(dy, dy, xx));"),
    ("wrong_axis_index", "float dy = a[1] - b[1];", "float dy = a[1] - b[0];"),
    ("sum_instead_of_difference", "float dx = a[0] - b[0];",
     "float dx = a[0] + b[0];"),
    ("fps_tie_to_larger_index", "if (m[j] > m[best]) best = j;",
     "if (m[j] >= m[best]) best = j;"),
    ("fps_ignores_start", "int64_t c = start_idx;", "int64_t c = 0;"),
    ("fps_no_min_update", "if (s < m[j]) m[j] = s;", "if (s > m[j]) m[j] = s;"),
    ("knn_tie_to_larger_index", "if (a->j < b->j) return -1;\n    if (a->j > b->j) return 1;",
     "if (a->j < b->j) return 1;\n    if (a->j > b->j) return -1;"),
    ("knn_returns_squared", "out_dist[r * k + t] = sqrtf(cand[t].s);",
     "out_dist[r * k + t] = cand[t].s;"),
    ("bq_non_strict", "if (s < R2) {", "if (s <= R2) {"),
    ("bq_radius_squared_in_double",
     "float r32 = (float)radius;\n    float r2 = r32 * r32;",
     "float r2 = (float)(radius * radius);"),
    ("bq_padding_zero_index", "out_idx[r * K + cnt] = -1;",
     "out_idx[r * K + cnt] = 0;"),
    ("bq_keeps_last_k", "for (int64_t j = 0; j < N && cnt < K; ++j) {\n            float s = orc_s32(q, x + 3 * j);\n            if (s < R2) {",
     "for (int64_t j = N - 1; j >= 0 && cnt < K; --j) {\n            float s = orc_s32(q, x + 3 * j);\n            if (s < R2) {"),
    ("bq_masked_non_strict", "int accept = s < R2;", "int accept = s <= R2;"),
    ("bq_masked_padding_zero_index", "out_idx[r * K + cnt] = (int64_t)-1;",
     "out_idx[r * K + cnt] = 0;"),
    ("lengths_ignored", "return len[b] > full ? full : len[b];", "return full;"),
    ("knn_masked_squared_flag_inverted",
     "squared ? cand[t].s : sqrtf(cand[t].s)", "squared ? sqrtf(cand[t].s) : cand[t].s"),
    ("bq_masked_rows_past_length_searched",
     "if (i < nq) {\n            const float *q = query + (size_t)row * 3;\n            const float *x = ref + (size_t)b * (size_t)N * 3;\n            for (int64_t j = 0; j < nr && cnt < K; ++j) {",
     "if (1) {\n            const float *q = query + (size_t)row * 3;\n            const float *x = ref + (size_t)b * (size_t)N * 3;\n            for (int64_t j = 0; j < nr && cnt < K; ++j) {"),
    ("gather_padding_not_zero", "o[0] = o[1] = o[2] = 0.0f;",
     "o[0] = x[b * N * 3]; o[1] = x[b * N * 3 + 1]; o[2] = x[b * N * 3 + 2];"),
    ("interp_wrong_weight_slot", "term[t] = wi[t] * v;", "term[t] = wi[0] * v;"),
    ("interp_padding_reads_feature_0", "float v = id[t] == -1 ? 0.0f : fr[id[t]];",
     "float v = id[t] == -1 ? fr[0] : fr[id[t]];"),
    ("interp_backward_drops_weight", "float p = w[(b * n + i) * 3 + t] * gi[i];",
     "float p = gi[i];"),
    ("interp_backward_overwrites", "gr[m] = gr[m] + p;", "gr[m] = p;"),
    ("knn_d_reversed_dimensions", "for (int64_t d = 0; d < D; ++d) {\n        float t = a[d] - b[d];",
     "for (int64_t d = D - 1; d >= 0; --d) {\n        float t = a[d] - b[d];"),
    ("knn_d_fma", "float t2 = t * t;\n        s = s + t2;", "s = fmaf(t, t, s);"),
    ("knn_d_drops_last_dimension", "for (int64_t d = 0; d < D; ++d) {\n        float t = a[d] - b[d];",
     "for (int64_t d = 0; d + 1 < D; ++d) {\n        float t = a[d] - b[d];"),
    ("knn_d_squared_ignored", "out_dist[r * k + t] = squared ? sd : sqrtf(sd);",
     "out_dist[r * k + t] = sqrtf(sd);"),
]

PIN_FUNCTIONS = [
    (pins.test_worked_example_fps, {}),
    (pins.test_worked_example_knn, {}),
    (pins.test_worked_example_ball_query, {}),
    (pins.test_s32_matches_exact_per_operation_rounding, {}),
    (pins.test_radius_threshold_is_float32_square_of_float32_radius, {}),
    (pins.test_ball_query_boundary_strict, {}),
    (pins.test_ball_query_threshold_not_double_square, {}),
    (pins.test_ball_query_k_equals_n_is_nonzero, {}),
    (pins.test_ball_query_first_k_in_input_order, {}),
    (pins.test_knn_matches_exact_sort, {"seed": 1, "grid": 1 / 8}),
    (pins.test_knn_duplicate_ties_go_to_smaller_index, {}),
    (pins.test_fps_line_matches_interval_bisection, {"n": 23, "start": 7}),
    (pins.test_fps_matches_brute_force, {"seed": 1, "grid": 1 / 4}),
    (pins.test_ball_query_scan_length, {}),
    (ext.test_quickstart_three_nn, {}),
    (ext.test_quickstart_three_interpolate, {}),
    (ext.test_quickstart_chamfer, {}),
    (ext.test_knn_masked_equals_knn_on_sliced_clouds, {}),
    (ext.test_knn_masked_squared_is_s32_of_the_pair, {}),
    (ext.test_ball_query_masked_equals_sliced, {}),
    (ext.test_gather_points_matches_fancy_indexing, {}),
    (ext.test_three_interpolate_one_hot_is_a_gather, {}),
    (ext.test_three_interpolate_exact_on_small_integers, {}),
    (ext.test_three_interpolate_padding_reads_zero, {}),
    (ext.test_three_interpolate_backward_exact_on_small_integers, {}),
    (ext.test_chamfer_brute_force_and_reductions, {}),
    (ext.test_chamfer_lengths_equal_sliced_clouds, {}),
    (kd.test_distance_matches_exact_rounding_per_operation, {}),
    (kd.test_order_of_accumulation_is_increasing_dimension, {}),
    (kd.test_three_dimensions_equal_the_point_operator, {}),
    (kd.test_selection_on_a_lattice_is_the_exact_lexsort, {}),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name, old, new):
    src = oracle_mod.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    lib = oracle_mod.compile_variant(src.replace(old, new),
                                     os.path.join(tmp_path, f"lib_{name}.so"))
    caught = []
    with oracle_mod.use_library(lib):
        for fn, kw in PIN_FUNCTIONS:
            try:
                fn(oracle_mod, **kw)
            except (AssertionError, ValueError):
                caught.append(fn.__name__)
            except pytest.skip.Exception:
                pass
    assert caught, f"no pin caught the planted mistake {name}"


def test_unmodified_copy_passes_every_pin(oracle_mod, tmp_path):
    lib = oracle_mod.compile_variant(oracle_mod.source_text(),
                                     os.path.join(tmp_path, "lib_same.so"))
    with oracle_mod.use_library(lib):
        for fn, kw in PIN_FUNCTIONS:
            fn(oracle_mod, **kw)
