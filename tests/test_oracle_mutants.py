"""Plant plausible mistakes in copies of the oracle and check the pins fail.

Each mutant is one textual edit of oracle/moe_oracle.c, compiled into a
scratch directory.  The pins of tests/test_oracle_pins.py are then run
against the mutant; at least one of them must fail.  The real oracle is
never modified.
"""
import os
import tempfile

import numpy as np
import pytest

import test_oracle_pins as pins
from oracle import build as obuild
from oracle import oracle as real

MUTANTS = {
    "combine_descending_rank": (
        "for (int d = 0; d < R; ++d) {\n                if (!(mask & (1u << d)))",
        "for (int d = R - 1; d >= 0; --d) {\n                if (!(mask & (1u << d)))"),
    "combine_drops_last_rank": (
        "for (int d = 0; d < R; ++d) {\n                if (!(mask & (1u << d)))",
        "for (int d = 0; d < R - 1; ++d) {\n                if (!(mask & (1u << d)))"),
    "weighted_uses_fma": (
        "float p = wd[(size_t)flat * R + d] * v;\n                    a = a + p;",
        "a = fmaf(wd[(size_t)flat * R + d], v, a);"),
    "weighted_ignores_weight": (
        "float p = wd[(size_t)flat * R + d] * v;",
        "float p = v;"),
    "residual_added_after_narrowing": (
        "hsum[h] = acc[h] + oracle_f32_from_bf16(",
        "hsum[h] = oracle_f32_from_bf16(oracle_bf16_from_f32(acc[h])) + oracle_f32_from_bf16("),
    "eps_outside_sqrt": (
        "1.0 / sqrt(sumsq / (double)H + (double)eps)",
        "1.0 / (sqrt(sumsq / (double)H) + (double)eps)"),
    "mean_over_h_minus_1": (
        "sumsq / (double)H + (double)eps",
        "sumsq / (double)(H - 1) + (double)eps"),
    "gamma_ignored": (
        "double y = (double)hsum[h] * inv * (double)oracle_f32_from_bf16(gamma[h]);",
        "double y = (double)hsum[h] * inv;"),
    "wd_sums_all_k": (
        "if (e / Epr == d)\n                        sum = sum + w[k];",
        "sum = sum + w[k];"),
    "no_nonlocal_id_masking": (
        "recv_ids[slot * K + k] = local ? e : -1;",
        "recv_ids[slot * K + k] = e;"),
    "slots_in_descending_token_order": (
        "for (int t = 0; t < T; ++t) {\n                size_t at",
        "for (int t = T - 1; t >= 0; --t) {\n                size_t at"),
    "narrowing_truncates": (
        "kept += 1u;",
        "kept += 0u;"),
    "local_counts_collapsed": (
        "local_expert_counts[d * Epr + (e - d * Epr)] += 1;",
        "local_expert_counts[d * Epr] += 1;"),
    "invalid_ids_not_counted": (
        "invalid += 1;",
        "invalid += 0;"),
    "tree_without_bf16_rounding": (
        "a[k] = oracle_f32_from_bf16(oracle_bf16_from_f32(a[k] + a[k + stride]));",
        "a[k] = a[k] + a[k + stride];"),
    "tree_keeps_duplicate_ranks": (
        "            if (!earlier)\n                slot_dest[k] = d;",
        "            (void)earlier;\n            slot_dest[k] = d;"),
    "tree_slots_in_rank_order": (
        "            int d = ids[k] / Epr;\n            int earlier = 0;",
        "            int d = (K - 1 - k) % R;\n            int earlier = 0;"),
    "fp8_truncates": (
        "    if (dropped > half || (dropped == half && (kept & 1u)))\n        kept += 1;",
        "    if (0)\n        kept += 1;"),
    "fp8_scale_for_wrong_format_max": (
        "float sc = amax > 0.0f ? amax / 448.0f : 1.0f;\n        scale[i] = sc;\n        for (int h = 0; h < H; ++h)\n            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(oracle_f32_from_bf16(",
        "float sc = amax > 0.0f ? amax / 240.0f : 1.0f;\n        scale[i] = sc;\n        for (int h = 0; h < H; ++h)\n            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(oracle_f32_from_bf16("),
    "fp8_overflow_to_nan": (
        "    if (exp32 == 0xffu || fabsf(f) > 448.0f)\n        return (uint8_t)(sign | 0x7e);",
        "    if (exp32 == 0xffu || fabsf(f) > 448.0f)\n        return (uint8_t)(sign | 0x7f);"),
    "experts_sources_descending": (
        "for (int s = 0; s < R; ++s) {\n        for (int t = 0; t < T; ++t) {\n            long flat",
        "for (int s = R - 1; s >= 0; --s) {\n        for (int t = 0; t < T; ++t) {\n            long flat"),
    "experts_duplicate_weights_not_summed": (
        "if (ids[k2] == e)\n                        sum = sum + w[k2];",
        "if (k2 == k)\n                        sum = sum + w[k2];"),
    "experts_duplicates_sent_twice": (
        "if (!first)\n                    continue;",
        "(void)first;"),
    "experts_combine_reverse_k": (
        "for (int k = 0; k < K; ++k) {\n                int32_t row = send_row",
        "for (int k = K - 1; k >= 0; --k) {\n                int32_t row = send_row"),
    "gemm_weights_transposed": (
        "const uint16_t *wr = w + ((size_t)e * N + n) * H;\n                double acc = 0.0;\n                for (int h = 0; h < H; ++h)\n                    acc += (double)oracle_f32_from_bf16(xr[h]) * (double)oracle_f32_from_bf16(wr[h]);",
        "const uint16_t *wr = w + (size_t)e * N * H;\n                double acc = 0.0;\n                for (int h = 0; h < H; ++h)\n                    acc += (double)oracle_f32_from_bf16(xr[h]) * (double)oracle_f32_from_bf16(wr[(size_t)h * N + n]);"),
    "gemm_wrong_expert_weights": (
        "const uint16_t *wr = w + ((size_t)e * N + n) * H;",
        "const uint16_t *wr = w + ((size_t)((e + 1) % E) * N + n) * H;"),
    "gemm_fp8_ignores_channel_scale": (
        "(double)sx[(size_t)e * cap + j] * (double)sw[(size_t)e * N + n] * acc;",
        "(double)sx[(size_t)e * cap + j] * acc;"),
    "fp8_f32_amax_without_fabs": (
        "if (fabsf(row[h]) > amax)\n                amax = fabsf(row[h]);",
        "if (row[h] > amax)\n                amax = row[h];"),
    "fp8_f32_quotient_multiplies": (
        "oracle_fp8e4m3_from_f32(row[h] / sc);",
        "oracle_fp8e4m3_from_f32(row[h] * sc);"),
    "fp8_f32_zero_row_scale_zero": (
        "float sc = amax > 0.0f ? amax / 448.0f : 1.0f;\n        scale[i] = sc;\n        for (int h = 0; h < H; ++h)\n            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(row[h] / sc);",
        "float sc = amax / 448.0f;\n        scale[i] = sc;\n        for (int h = 0; h < H; ++h)\n            q[(size_t)i * H + h] = oracle_fp8e4m3_from_f32(row[h] / sc);"),
    "gemm_rank_descending_k": (
        "for (int k = 0; k < K; ++k) {\n                int e = ids[k];\n                if (e < 0)\n                    continue;\n                const uint16_t *wr",
        "for (int k = K - 1; k >= 0; --k) {\n                int e = ids[k];\n                if (e < 0)\n                    continue;\n                const uint16_t *wr"),
    "gemm_rank_gates_ignored": (
        "float gk = apply_gates ? g[k] : 1.0f;",
        "float gk = 1.0f;"),
    "gemm_rank_uses_fma": (
        "float p = gk * yk;\n                a = a + p;",
        "a = fmaf(gk, yk, a);"),
    "gemm_rank_expert_output_not_narrowed": (
        "float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));",
        "float yk = (float)y;"),
    "gemm_rank_wrong_expert_weights": (
        "const uint16_t *wr = w + ((size_t)e * N + n) * H;\n                double y = 0.0, mag = 0.0;",
        "const uint16_t *wr = w + ((size_t)(e ^ 1) * N + n) * H;\n                double y = 0.0, mag = 0.0;"),
    "gemm_rank_fp8_ignores_row_scale": (
        "const double scale = sx * (double)sw[(size_t)e * N + n];",
        "const double scale = (double)sw[(size_t)e * N + n];"),
    "gemm_rank_fp8_ignores_channel_scale": (
        "const double scale = sx * (double)sw[(size_t)e * N + n];",
        "const double scale = sx;"),
    "gemm_rank_fp8_next_row_scale": (
        "const double sx = (double)recv_scale[flat];",
        "const double sx = (double)recv_scale[(flat + 1) % ((long)R * R * m)];"),
    "gemm_rank_fp8_descending_k": (
        "for (int k = 0; k < K; ++k) {\n                int e = ids[k];\n                if (e < 0)\n                    continue;\n                const uint8_t *wr",
        "for (int k = K - 1; k >= 0; --k) {\n                int e = ids[k];\n                if (e < 0)\n                    continue;\n                const uint8_t *wr"),
    "gemm_rank_fp8_expert_output_not_narrowed": (
        "double y = scale * acc;\n                float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));",
        "double y = scale * acc;\n                float yk = (float)y;"),
    "gemm_rank_fp8_gates_ignored": (
        "double y = scale * acc;\n                float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));\n                float gk = apply_gates ? g[k] : 1.0f;",
        "double y = scale * acc;\n                float yk = oracle_f32_from_bf16(oracle_bf16_from_f32((float)y));\n                float gk = 1.0f;"),
    "gemm_rank_fp8_uses_fma": (
        "float gk = apply_gates ? g[k] : 1.0f;\n                float p = gk * yk;\n                a = a + p;\n                ym += fabs((double)gk) * fabs(y);\n                sm += fabs((double)gk) * fabs(scale) * mag;",
        "float gk = apply_gates ? g[k] : 1.0f;\n                a = fmaf(gk, yk, a);\n                ym += fabs((double)gk) * fabs(y);\n                sm += fabs((double)gk) * fabs(scale) * mag;"),
    "gemm_rank_fp8_wrong_expert_weights": (
        "const uint8_t *wr = qw + ((size_t)e * N + n) * H;\n                const double scale",
        "const uint8_t *wr = qw + ((size_t)(e ^ 1) * N + n) * H;\n                const double scale"),
    "gemm_rank_fp8_weights_transposed": (
        "double prod = (double)oracle_f32_from_fp8e4m3(xr[h]) *\n                                  (double)oracle_f32_from_fp8e4m3(wr[h]);",
        "double prod = (double)oracle_f32_from_fp8e4m3(xr[h]) *\n                                  (double)oracle_f32_from_fp8e4m3(qw[(size_t)e * N * H + (size_t)(h % N) * H + n % H]);"),
    "gemm_rank_fp8_reads_first_row_of_plane": (
        "const uint8_t *xr = recv_x8 + (size_t)flat * H;",
        "const uint8_t *xr = recv_x8 + (size_t)(flat - j) * H;"),
    "dispatch_copies_wrong_source_token": (
        "const uint16_t *row = x + ((size_t)s * T + t) * H;",
        "const uint16_t *row = x + ((size_t)s * T + (t + 1) % T) * H;"),
}


class MutantOracle:
    """The numpy front end bound to a mutant library."""

    def __init__(self, handle):
        self.h = handle

    def lib(self):
        return self.h

    def bf16_bits(self, v):
        return real.bf16_bits(v, handle=self.h)

    def route(self, *a, **k):
        return real.route(*a, handle=self.h, **k)

    def dispatch(self, *a, **k):
        return real.dispatch(*a, handle=self.h, **k)

    def combine(self, *a, **k):
        return real.combine(*a, handle=self.h, **k)

    def combine_topk_tree(self, *a, **k):
        return real.combine_topk_tree(*a, handle=self.h, **k)

    def route_experts(self, *a, **k):
        return real.route_experts(*a, handle=self.h, **k)

    def dispatch_experts(self, *a, **k):
        return real.dispatch_experts(*a, handle=self.h, **k)

    def combine_experts(self, *a, **k):
        return real.combine_experts(*a, handle=self.h, **k)

    def expert_gemm(self, *a, **k):
        return real.expert_gemm(*a, handle=self.h, **k)

    def expert_gemm_rank(self, *a, **k):
        return real.expert_gemm_rank(*a, handle=self.h, **k)

    def expert_gemm_rank_fp8(self, *a, **k):
        return real.expert_gemm_rank_fp8(*a, handle=self.h, **k)

    def expert_gemm_fp8(self, *a, **k):
        return real.expert_gemm_fp8(*a, handle=self.h, **k)

    def quantize_f32_rows_fp8(self, x):
        return real.quantize_f32_rows_fp8(x, handle=self.h)

    def fp8_bits(self, v):
        return real.fp8_bits(v, handle=self.h)

    def fp8_to_f32(self, v):
        return real.fp8_to_f32(v, handle=self.h)

    def quantize_rows_fp8(self, x):
        return real.quantize_rows_fp8(x, handle=self.h)


PIN_TESTS = [
    (pins.test_bf16_rounding_matches_library_routine, {}),
    (pins.test_probe_pow2_rank_sum_is_255, {}),
    (pins.test_probe_reduction_discriminator, {}),
    (pins.test_probe_slot_order_is_ascending_token, {}),
    (pins.test_probe_partial_routing_and_duplicates, {}),
    (pins.test_route_brute_force, {"seed": 3}),
    (pins.test_route_brute_force, {"seed": 0}),
    (pins.test_dispatch_payload_identity, {}),
    (pins.test_identity_unweighted_is_n_times_x, {}),
    (pins.test_identity_weighted_dyadic_returns_x_once, {}),
    (pins.test_weighted_sum_within_fp32_error_bound, {}),
    (pins.test_ascending_rank_order_closed_form, {}),
    (pins.test_weighted_product_is_not_fused, {}),
    (pins.test_residual_add_uses_fp32_sum, {}),
    (pins.test_rmsnorm_constant_row_closed_form, {"cval": 1e-3}),
    (pins.test_rmsnorm_matches_library_routine, {}),
    (pins.test_probe_topk_tree_gives_the_pages_bf16_tree_value, {}),
    (pins.test_topk_tree_blanks_duplicate_ranks, {}),
    (pins.test_topk_tree_keeps_top_k_slot_order, {}),
    (pins.test_fp8_narrowing_matches_library_routine, {}),
    (pins.test_fp8_saturates_and_keeps_nan, {}),
    (pins.test_fp8_row_scaling_closed_forms, {}),
    (pins.test_fp8_round_trip_within_format_bound, {}),
    (pins.test_fp8_f32_rows_closed_forms, {}),
    (pins.test_fp8_f32_rows_match_library_cast, {}),
    (pins.test_fp8_f32_rows_round_trip_over_the_binary32_range, {}),
    (pins.test_route_experts_brute_force, {"seed": 1}),
    (pins.test_expert_dispatch_payload_identity, {}),
    (pins.test_expert_identity_unweighted_counts_distinct_experts, {}),
    (pins.test_expert_identity_weighted_sums_duplicate_weights, {}),
    (pins.test_expert_combine_sums_in_problem_order, {}),
    (pins.test_expert_gemm_identity_and_power_of_two_weights, {}),
    (pins.test_expert_gemm_matches_library_matmul, {}),
    (pins.test_expert_gemm_fp8_identity_and_library_matmul, {}),
    (pins.test_expert_gemm_rank_identity_weights_count_local_experts, {}),
    (pins.test_expert_gemm_rank_power_of_two_weights_and_dyadic_gates, {}),
    (pins.test_expert_gemm_rank_matches_library_matmul_and_gate_order, {}),
    (pins.test_expert_gemm_rank_equals_expert_layout_with_one_expert_per_rank, {}),
    (pins.test_expert_gemm_rank_sums_in_top_k_order, {}),
    (pins.test_expert_gemm_rank_fp8_identity_codes_count_local_experts, {}),
    (pins.test_expert_gemm_rank_fp8_matches_library_matmul_and_gate_order, {}),
    (pins.test_expert_gemm_rank_fp8_equals_expert_layout_with_one_expert_per_rank, {}),
    (pins.test_expert_gemm_rank_fp8_sums_in_top_k_order, {}),
    (pins.test_expert_gemm_rank_fp8_row_list_matches_full, {}),
    (pins.test_expert_gemm_rank_fp8_gate_product_is_not_fused, {}),
]


def _compile_mutant(name, tmpdir):
    """Apply the edit at its first occurrence (for the epilogue lines, which
    oracle_combine and oracle_combine_topk_tree share, that is oracle_combine)."""
    old, new = MUTANTS[name]
    src = open(obuild.SOURCE).read()
    assert src.count(old) >= 1, "mutation site for %s not found" % name
    path = os.path.join(tmpdir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    return obuild.build(force=True, source=path, output=os.path.join(tmpdir, name + ".so"))


def test_pins_pass_on_real_oracle():
    o = MutantOracle(real.lib())
    for fn, kw in PIN_TESTS:
        fn(o, **kw)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    with tempfile.TemporaryDirectory() as tmp:
        o = MutantOracle(real.lib(_compile_mutant(name, tmp)))
        caught = []
        for fn, kw in PIN_TESTS:
            try:
                fn(o, **kw)
            except AssertionError:
                caught.append(fn.__name__)
        assert caught, "no pin caught mutant %s" % name
