"""The pins catch plausible mistakes in the oracle.

Each case copies ``oracle/oracle.c``, plants one mistake by a textual
replacement (a dropped term, a wrong exponent, a misplaced epsilon, a
transposed operand, a wrong region order...), compiles the copy on the CPU
and runs every pin against it: at least one pin must fail.  The oracle
itself is never modified.
"""

import pytest

import oracle as oracle_pkg
from oracle_pins import PINS

MUTANTS = {
    "no_bias_correction_1": ("m_t / (1.0 - pow(beta1, (double)t))", "m_t"),
    "no_bias_correction_2": ("v_t / (1.0 - pow(beta2, (double)t))", "v_t"),
    "bias_exponent_t_plus_1": ("pow(beta1, (double)t)", "pow(beta1, (double)(t + 1))"),
    "bias_exponent_t_minus_1": ("pow(beta2, (double)t)", "pow(beta2, (double)(t - 1))"),
    "eps_inside_sqrt": ("lr * m_hat / (sqrt(v_hat) + eps)", "lr * m_hat / sqrt(v_hat + eps)"),
    "uncorrected_v_in_denominator": ("lr * m_hat / (sqrt(v_hat) + eps)",
                                     "lr * m_hat / (sqrt(v_t) + eps)"),
    "decay_after_update": ("out->w = w_decayed - update;",
                           "out->w = (w - update) * (1.0 - lr * wd);"),
    "coupled_l2_decay": ("double g_hat = g * s;", "double g_hat = g * s + wd * w;"),
    "no_decay": ("w * (1.0 - lr * wd)", "w"),
    "decay_without_lr": ("w * (1.0 - lr * wd)", "w * (1.0 - wd)"),
    "update_sign": ("out->w = w_decayed - update;", "out->w = w_decayed + update;"),
    "swapped_betas": ("beta1 * m + (1.0 - beta1) * g_hat",
                      "beta2 * m + (1.0 - beta2) * g_hat"),
    "m_from_unclipped": ("(1.0 - beta1) * g_hat", "(1.0 - beta1) * g"),
    "v_from_unclipped": ("(g_hat * g_hat)", "(g * g)"),
    "v_not_squared": ("(g_hat * g_hat)", "(g_hat)"),
    "m_weights_swapped": ("beta1 * m + (1.0 - beta1) * g_hat",
                          "(1.0 - beta1) * m + beta1 * g_hat"),
    "always_clip": ("if (norm > c)", "if (norm > 0.0)"),
    "never_clip": ("if (norm > c)", "if (0)"),
    "clip_factor_inverted": ("return c / norm;", "return norm / c;"),
    "clip_with_epsilon": ("return c / norm;", "return c / (norm + 1e-6);"),
    "norm_abs_sum": ("s = s + x * x;", "s = s + fabs(x);"),
    "norm_no_sqrt": ("return sqrt(oracle_sumsq(g, n));", "return oracle_sumsq(g, n);"),
    "norm_skips_last": ("for (int64_t i = 0; i < n; ++i) {\n        double x",
                        "for (int64_t i = 0; i + 1 < n; ++i) {\n        double x"),
    "nonfinite_not_detected": ("if (!isfinite(norm))\n        return OR_ENONFINITE;", ""),
    "header_order_swapped": ("put_le32(out, (uint32_t)step);\n    put_le32(out + 4, (uint32_t)n);",
                             "put_le32(out, (uint32_t)n);\n    put_le32(out + 4, (uint32_t)step);"),
    "pack_m_v_swapped": ("memcpy(out + 8 + bytes, m, bytes);\n    memcpy(out + 8 + 2 * bytes, v, bytes);",
                         "memcpy(out + 8 + bytes, v, bytes);\n    memcpy(out + 8 + 2 * bytes, m, bytes);"),
    "file_m_v_swapped": ("rc = write_all(f, m, bytes);\n    if (rc == OR_OK)\n        rc = write_all(f, v, bytes);",
                         "rc = write_all(f, v, bytes);\n    if (rc == OR_OK)\n        rc = write_all(f, m, bytes);"),
    "file_header_big_endian": ("put_le32(header, (uint32_t)step);",
                               "put_le32(header, __builtin_bswap32((uint32_t)step));"),
    "no_rename_tmp_left": ("if (rename(tmp_path, final_path) != 0) {",
                           "if (link(tmp_path, final_path) != 0) {"),
    "name_without_padding": ("\"%s/step_%06d.bin\"", "\"%s/step_%d.bin\""),
    "reader_no_size_check": ("if ((int64_t)st.st_size != oracle_ckpt_size(n)) {", "if (0) {"),
    "reader_no_n_check": ("if (n != n_expected) {", "if (0) {"),
    "reader_accepts_negative": ("if (step < 0 || n < 0) {", "if (0) {"),
    "reader_m_v_swapped": ("fread(m, 1, bytes, f) != bytes ||\n        fread(v, 1, bytes, f) != bytes",
                           "fread(v, 1, bytes, f) != bytes ||\n        fread(m, 1, bytes, f) != bytes"),
    "step_rounds_m_from_v": ("m[i] = (float)r.m;", "m[i] = (float)r.v;"),
    "step_t_off_by_one": ("double s = oracle_clip_scale(norm, clip);",
                          "double s = oracle_clip_scale(norm, clip);\n    t = t + 1;"),
    "tensor_sum_skips_last": ("out[k] = oracle_sumsq(g + offsets[k], numels[k]);",
                              "out[k] = oracle_sumsq(g + offsets[k], numels[k] - 1);"),
    "tensor_sum_shifted": ("out[k] = oracle_sumsq(g + offsets[k], numels[k]);",
                           "out[k] = oracle_sumsq(g + offsets[k] + 1, numels[k]);"),
    "bf16_decode_shift": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;"),
    "f16_decode_bias": ("mag = ldexp((double)(1024 + frac), ex - 25);",
                        "mag = ldexp((double)(1024 + frac), ex - 24);"),
    "f16_no_subnormal_scale": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    "bf16_round_half_up": ("return (uint16_t)((bits + 0x7fffu + lsb) >> 16);",
                           "return (uint16_t)((bits + 0x8000u) >> 16);"),
    "f16_ties_away": ("if (rem > 0.5 || (rem == 0.5 && (k & 1u)))", "if (rem >= 0.5)"),
    "f16_overflow_never": ("if (a >= 65520.0)", "if (a >= 1e300)"),
    "mixed_ignores_scale": ("double x = gi * grad_scale;", "double x = gi;"),
    "scaled_clip_on_raw_norm": ("double x = (double)g[i] * grad_scale;\n        sumsq = sumsq + x * x;",
                                "double x = (double)g[i];\n        sumsq = sumsq + x * x;"),
    "scaled_update_unscaled": ("oracle_adamw_element((double)w[i], (double)g[i] * grad_scale,",
                               "oracle_adamw_element((double)w[i], (double)g[i],"),
    "range_starts_late": ("for (int64_t j = lo; j < hi; ++j) {", "for (int64_t j = lo + 1; j < hi; ++j) {"),
    "range_gradient_shifted": ("oracle_adamw_element((double)w[j], (double)g[j],",
                               "oracle_adamw_element((double)w[j], (double)g[j + (j + 1 < hi)],"),
    "mask_ignored": ("double wd_k = decay[k] ? wd : 0.0;", "double wd_k = wd;"),
    "mask_inverted": ("double wd_k = decay[k] ? wd : 0.0;", "double wd_k = decay[k] ? 0.0 : wd;"),
    "mask_shifted": ("double wd_k = decay[k] ? wd : 0.0;",
                     "double wd_k = decay[k + 1 < n_tensors ? k + 1 : k] ? wd : 0.0;"),
    "mask_skips_exempt_update": ("double wd_k = decay[k] ? wd : 0.0;",
                                 "double wd_k = decay[k] ? wd : 0.0;\n        if (!decay[k]) continue;"),
    "mask_range_short": ("i < offsets[k] + numels[k]; ++i)", "i + 1 < offsets[k] + numels[k]; ++i)"),
    "mask_no_table_check": ("if (offsets[k] != next || numels[k] < 0)", "if (numels[k] < 0)"),
    "scaled_twice": ("double x = (double)g[i] * grad_scale;",
                     "double x = (double)g[i] * grad_scale * grad_scale;"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle_pkg.SOURCE) as f:
        return f.read()


def _pins_fail(o, tmp_path):
    failures = []
    for pin in PINS:
        d = tmp_path / pin.__name__
        d.mkdir()
        try:
            pin(o, d)
        except Exception as e:  # noqa: BLE001 - any failure counts
            failures.append((pin.__name__, type(e).__name__))
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    # planted wherever the anchor occurs (the same mistake made consistently)
    assert source.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = str(tmp_path / "mutant.so")
    oracle_pkg.build(str(src), lib)
    failures = _pins_fail(oracle_pkg.Oracle(lib), tmp_path)
    assert failures, f"no pin caught mutant {name}"


def test_unmutated_copy_passes(source, tmp_path):
    src = tmp_path / "copy.c"
    src.write_text(source)
    lib = str(tmp_path / "copy.so")
    oracle_pkg.build(str(src), lib)
    assert _pins_fail(oracle_pkg.Oracle(lib), tmp_path) == []
