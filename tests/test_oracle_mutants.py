"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant below is a plausible slip (a dropped term, a wrong sign, a wrong
index, a transposed operand, a dropped partial block, a missing absolute
value, a missing initialisation).  The mistake is planted in a private copy
of the C source, compiled on the CPU and run against the pin suite; all
mutants keep every memory access inside the caller's arrays.
"""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "q8mv_oracle.c")

MUTANTS = {
    "scale_row_mod": ("const float *s_row = S + (k / Q8MV_ORACLE_BLK) * N;",
                      "const float *s_row = S + ((k % Q8MV_ORACLE_BLK) % ((K + 31) / 32)) * N;"),
    "scale_row_64": ("const float *s_row = S + (k / Q8MV_ORACLE_BLK) * N;",
                     "const float *s_row = S + (k / 64) * N;"),
    "factored_prev_scale_row": ("const float *s_row = S + b * N;",
                                "const float *s_row = S + (b > 0 ? b - 1 : 0) * N;"),
    "drop_partial_block": ("return (K + Q8MV_ORACLE_BLK - 1) / Q8MV_ORACLE_BLK;",
                           "return K / Q8MV_ORACLE_BLK;"),
    "drop_first_row_of_block": ("for (int64_t k = k_begin; k < k_end; ++k) {\n            const double a = (double)A[k];\n            const int8_t *w_row = W + k * N;\n            for (int64_t n = 0; n < N; ++n) {\n                const double aw",
                                "for (int64_t k = k_begin + 1; k < k_end; ++k) {\n            const double a = (double)A[k];\n            const int8_t *w_row = W + k * N;\n            for (int64_t n = 0; n < N; ++n) {\n                const double aw"),
    "wrong_sign": ("C[n] += part[n] * s;", "C[n] -= part[n] * s;"),
    "transposed_w_factored": ("const double aw = a * (double)w_row[n];",
                              "const double aw = a * (double)W[n * K + k];"),
    "transposed_w_unfactored": ("C[n] += a * (double)w_row[n] * (double)s_row[n];",
                                "C[n] += a * (double)W[n * K + k] * (double)s_row[n];"),
    "bound_without_abs": ("mag[n] += fabs(aw);", "mag[n] += aw;"),
    "unsigned_bytes": ("const double aw = a * (double)w_row[n];",
                       "const double aw = a * (double)(uint8_t)w_row[n];"),
    "no_zero_init": ("        C[n] = 0.0;\n        if (bound) bound[n] = 0.0;",
                     "        if (bound) bound[n] = 0.0;"),
    "block_sums_missing_mask": ("        if (k_end > K) k_end = K;\n        for (int64_t k = k_begin; k < k_end; ++k) {\n            const double a = (double)A[k];\n            const int8_t *w_row = W + k * N;\n            for (int64_t n = 0; n < N; ++n) p_row[n] += a * (double)w_row[n];",
                                "        if (k_end > K) k_end = K;\n        for (int64_t k = k_begin; k < k_end; ++k) {\n            const double a = (double)A[k];\n            const int8_t *w_row = W + k * N;\n            for (int64_t n = 0; n < N; ++n) p_row[n] += a * (double)w_row[n] * (k + 1 < k_end);"),
    "batched_row_stride_n": ("q8mv_oracle_factored(K, N, A + m * K, W, S, C + m * N, bound ? bound + m * N : NULL)",
                             "q8mv_oracle_factored(K, N, A + m * (N < K ? N : K), W, S, C + m * N, bound ? bound + m * N : NULL)"),
    "batched_first_row_only": ("q8mv_oracle_factored(K, N, A + m * K, W, S, C + m * N, bound ? bound + m * N : NULL)",
                               "q8mv_oracle_factored(K, N, A, W, S, C + m * N, bound ? bound + m * N : NULL)"),
    "batched_rows_reversed": ("q8mv_oracle_factored(K, N, A + m * K, W, S, C + m * N, bound ? bound + m * N : NULL)",
                              "q8mv_oracle_factored(K, N, A + (M - 1 - m) * K, W, S, C + m * N, bound ? bound + m * N : NULL)"),
    "batched_skip_last_row": ("for (int64_t m = 0; m < M; ++m) {\n        const int rc",
                              "for (int64_t m = 0; m + 1 < M; ++m) {\n        const int rc"),
    "epi_bias_by_row": ("const double b = bias ? (double)bias[n] : 0.0;",
                        "const double b = bias ? (double)bias[m % N] : 0.0;"),
    "epi_residual_by_column": ("const double r = residual ? (double)residual[i] : 0.0;",
                               "const double r = residual ? (double)residual[n] : 0.0;"),
    "epi_beta_ignored": ("const double bc = beta != 0.0 ? beta * (double)c_old[i] : 0.0;",
                         "const double bc = 0.0;"),
    "epi_silu_sign": ("y = y / (1.0 + exp(-y));", "y = y / (1.0 + exp(y));"),
    "epi_gelu_cubic": ("(y + 0.044715 * y * y * y)", "(y + 0.0044715 * y * y * y)"),
    "epi_relu_leaky": ("y = y > 0.0 ? y : 0.0;", "y = y > 0.0 ? y : 0.01 * y;"),
    "epi_residual_dropped": ("out[i] = y + r;", "out[i] = y;"),
    "epi_alpha_ignored": ("const double ax = alpha * x[i];", "const double ax = x[i];"),
    "t_row_stride": ("const int8_t *w_row = Wt + n * K;", "const int8_t *w_row = Wt + n * (K > 1 ? K - 1 : K);"),
    "t_scale_row_of_next_output": ("const float *s_row = St + n * KB;",
                                   "const float *s_row = St + ((n + 1) % N) * KB;"),
    "t_scale_by_k_not_block": ("const double s = (double)s_row[b];",
                               "const double s = (double)s_row[b == 0 ? 0 : b - 1];"),
    "t_drop_masked_rows": ("            if (k_end > K) k_end = K;\n            double part = 0.0, part_mag = 0.0;",
                           "            if (k_end > K) k_end = k_begin;\n            double part = 0.0, part_mag = 0.0;"),
    "qa_no_abs": ("const float a = fabsf(A[k]);", "const float a = A[k];"),
    "qa_d_by_128": ("const float db = amax / 127.0f;", "const float db = amax / 128.0f;"),
    "qa_truncate": ("float r = rintf(x);", "float r = truncf(x);"),
    "qa_round_half_away": ("float r = rintf(x);", "float r = roundf(x);"),
    "i8_next_scale": ("const double scale = (double)d[b] * (double)St[n * KB + b];",
                      "const double scale = (double)d[b] * (double)St[n * KB + (b + 1) % KB];"),
    "i8_unsigned_codes": ("const int64_t p = (int64_t)q[k] * (int64_t)Wt[n * K + k];",
                          "const int64_t p = (int64_t)(uint8_t)q[k] * (int64_t)Wt[n * K + k];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.build(str(mutated), str(tmp_path / "libmutant.so"), force=True)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError) as e:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
