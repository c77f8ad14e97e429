"""Plant plausible mistakes in copies of the oracle (on the CPU only) and check
that the pins in ``test_oracle_pins.py`` catch every one of them.

Each mutant replaces one line of ``oracle/pkv_oracle.c`` in a temporary copy,
compiles it with the oracle's own flags and runs the whole battery of pins
against it; at least one pin must fail.  The real oracle is never modified.
"""
import os
import tempfile

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTANTS = {
    "sink_multiplied_by_scale": (
        "if (a->sinks) den += exp((double)a->sinks[h] - M);",
        "if (a->sinks) den += exp(a->scale * (double)a->sinks[h] - M);"),
    "slot_off_by_one": (
        "const int slot = j % P;",
        "const int slot = (j + 1) % P;"),
    "logical_page_off_by_one": (
        "const int32_t page = a->bt[(int64_t)b * a->bt_sb + j / P];\n        const int slot",
        "const int32_t page = a->bt[(int64_t)b * a->bt_sb + (j + P - 1) / P];\n        const int slot"),
    "window_off_by_one": (
        "if (a->window > 0 && L > a->window) s = L - a->window;",
        "if (a->window > 0 && L > a->window) s = L - a->window + 1;"),
    "gqa_lse_drops_max": (
        "    *lse = M + log(Z);\n    free(x); free(qd); free(vrow);",
        "    *lse = log(Z);\n    free(x); free(qd); free(vrow);"),
    "v_read_from_k_half": (
        "vrow[j - s] = krow + D;",
        "vrow[j - s] = krow;"),
    "kv_head_mapping_modulo": (
        "const int g = h / (a->Hq / a->Hkv);",
        "const int g = h % a->Hkv;"),
    "softmax_sign_flipped": (
        "for (int i = 0; i < n; ++i) Z += exp(x[i] - M);",
        "for (int i = 0; i < n; ++i) Z += exp(M - x[i]);"),
    "scale_dropped": (
        "x[j - s] = a->scale * dot;",
        "x[j - s] = dot;"),
    "empty_row_lse_zero": (
        "    if (n == 0) {\n        *lse = -INFINITY;",
        "    if (n == 0) {\n        *lse = 0.0;"),
    "mla_row_limit_off_by_one": (
        "int lim = L - a->qlen + 1 + t;",
        "int lim = L - a->qlen + t;"),
    "mla_real_seq_lens_ignored": (
        "if (Lr < lim) lim = Lr;",
        "(void)Lr;"),
    "mla_v_from_trailing_dims": (
        "out[d] += w * cache_elem(a, kbase[j] + d);",
        "out[d] += w * cache_elem(a, kbase[j] + (Lk - Lv) + d);"),
    "mla_k_scale_dropped": (
        "if (a->fp8) return pkv_oracle_e4m3_to_f64(a->cache[idx]) * a->k_scale;",
        "if (a->fp8) return pkv_oracle_e4m3_to_f64(a->cache[idx]);"),
    "e4m3_bias_8": (
        "v = ldexp(1.0 + (double)m / 8.0, e - 7);",
        "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal_exponent": (
        "v = ldexp((double)m / 8.0, -6);",
        "v = ldexp((double)m / 8.0, -7);"),
}

# (pin, kwargs) pairs: every non-parametrised pin and one instance of each
# parametrised one.
BATTERY = [
    (pins.test_e4m3_decode_matches_torch_all_codes, {}),
    (pins.test_block_table_worked_example, dict(Hq=8, Hkv=1)),
    (pins.test_oracle_matches_dense_scipy,
     dict(seed=1, B=3, Hq=8, Hkv=1, P=16, Lmax=64, sinks=True, window=0)),
    (pins.test_oracle_matches_dense_scipy,
     dict(seed=2, B=2, Hq=16, Hkv=2, P=32, Lmax=64, sinks=True, window=0)),
    (pins.test_oracle_matches_dense_scipy,
     dict(seed=4, B=3, Hq=8, Hkv=1, P=4, Lmax=40, sinks=True, window=7)),
    (pins.test_oracle_random_block_table_matches_dense, {}),
    (pins.test_single_key_returns_v_exactly, {}),
    (pins.test_constant_v_returns_constant, {}),
    (pins.test_empty_rows_write_zero_and_neg_inf_lse, {}),
    (pins.test_sink_limits, {}),
    (pins.test_window_equals_full_attention_on_last_w_keys, {}),
    (pins.test_head_grouping_uses_kv_head_h_div_group, {}),
    (pins.test_mla_qlen1_equals_dense_attention, dict(fp8=True)),
    (pins.test_mla_qlen1_equals_dense_attention, dict(fp8=False)),
    (pins.test_mla_verify_row_limits,
     dict(L=[10], real=[8], qlen=4, lims=[7, 8, 8, 8])),
    (pins.test_mla_verify_row_limits,
     dict(L=[40, 5], real=[37, 0], qlen=3, lims=[37, 37, 37, 0, 0, 0])),
    (pins.test_mla_v_is_the_leading_lv_dims_of_k, {}),
    (pins.test_mla_fp8_k_scale_scales_v_and_scores, {}),
]


def _build_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur exactly once"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.load(oracle.compile_oracle(path, os.path.join(tmp, f"lib{name}.so")))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(name, tmp)
        monkeypatch.setattr(pins, "LIB", lib)
        caught = []
        for fn, kw in BATTERY:
            try:
                if fn is pins.test_e4m3_decode_matches_torch_all_codes:
                    fn(lib)
                else:
                    fn(**kw)
            except (AssertionError, oracle.OracleError):
                caught.append(fn.__name__)
        assert caught, f"no pin catches mutant {name}"


def test_unmutated_oracle_passes_the_battery(monkeypatch):
    monkeypatch.setattr(pins, "LIB", None)
    for fn, kw in BATTERY:
        if fn is pins.test_e4m3_decode_matches_torch_all_codes:
            fn(oracle.load())
        else:
            fn(**kw)


# ---- paged KV append and the e4m3 encoder --------------------------------
import tests.test_oracle_append_pins as apins  # noqa: E402

APPEND_MUTANTS = {
    "append_position_is_seq_len": (
        "if (!append_slot(bt, bt_sb, max_blocks, num_blocks, b, L - 1, page_size, &blk, &slot)) {",
        "if (!append_slot(bt, bt_sb, max_blocks, num_blocks, b, L, page_size, &blk, &slot)) {"),
    "append_slot_off_by_one": (
        "    *slot = pos % page_size;",
        "    *slot = (pos + 1) % page_size;"),
    "mla_append_row_position": (
        "const int64_t pos = (int64_t)seq_lens[b] - qlen + t;",
        "const int64_t pos = (int64_t)seq_lens[b] - qlen + t + 1;"),
    "append_writes_unassigned_pages": (
        "    if (id < 0 || id >= num_blocks) return 0;",
        "    if (id >= num_blocks) return 0;"),
    "e4m3_encode_ties_away": (
        "        double q = rint(16.0 * f);     /* 8 * (2f): 8 .. 16 */",
        "        double q = round(16.0 * f);    /* 8 * (2f): 8 .. 16 */"),
    "e4m3_encode_no_saturation": (
        "        if (E > 8 || (E == 8 && q > 14.0)) { /* beyond 448: saturate */",
        "        if (E > 9) { /* beyond 448: saturate */"),
    "e4m3_encode_subnormal_step": (
        "        const double q = rint(a * 512.0); /* multiples of 2^-9: 0 .. 8 */",
        "        const double q = rint(a * 256.0); /* multiples of 2^-9: 0 .. 8 */"),
    "fp8_append_multiplies_by_k_scale": (
        "pkv_oracle_f32_to_e4m3(x / k_scale);",
        "pkv_oracle_f32_to_e4m3(x * k_scale);"),
}

APPEND_BATTERY = [
    (apins.test_gqa_append_worked_example, {}),
    (apins.test_mla_append_worked_example, dict(qlen=1)),
    (apins.test_mla_append_worked_example, dict(qlen=2)),
    (apins.test_append_skips_rows_without_a_position_or_page, {}),
    (apins.test_e4m3_encode_round_trips_every_code, {}),
    (apins.test_e4m3_encode_ties_to_even_and_saturates, {}),
    (apins.test_e4m3_encode_matches_torch_in_range, {}),
    (apins.test_mla_fp8_append_stores_e4m3_of_x_over_k_scale, {}),
]


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(name, monkeypatch):
    old, new = APPEND_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.compile_oracle(path, os.path.join(tmp, f"lib{name}.so")))
        monkeypatch.setattr(apins, "LIB", lib)
        caught = []
        for fn, kw in APPEND_BATTERY:
            try:
                fn(**kw)
            except (AssertionError, oracle.OracleError):
                caught.append(fn.__name__)
        assert caught, f"no pin catches mutant {name}"


# ---- the native-FP8 MLA query quantisation --------------------------------
import tests.test_oracle_q8_pins as qpins  # noqa: E402

Q8_MUTANTS = {
    "q8_scale_divisor": (
        "const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;",
        "const float sc = amax > 0.0f ? amax / 447.0f : 1.0f;"),
    "q8_absmax_signed": (
        "const float v = (float)fabs(pkv_oracle_bf16_to_f64(row[d]));",
        "const float v = (float)pkv_oracle_bf16_to_f64(row[d]);"),
    "q8_scale_ignored_by_verify": (
        "const double sq = (double)a->q8_scale[r * a->qs_sr + h];",
        "const double sq = 1.0;"),
    "q8_head_stride_ignored": (
        "const uint8_t *c8 = a->q8 + r * a->q8_sr + (int64_t)h * a->q8_sh;",
        "const uint8_t *c8 = a->q8 + r * a->q8_sr;"),
}

Q8_BATTERY = [
    (qpins.test_quantize_scale_is_absmax_over_448_in_fp32, {}),
    (qpins.test_quantize_absmax_element_is_448, {}),
    (qpins.test_quantize_zero_row_and_single_value, {}),
    (qpins.test_quantize_matches_torch_float8_conversion_below_the_max, {}),
    (qpins.test_quantize_error_within_half_a_step, {}),
    (qpins.test_verify_q8_equals_verify_for_exactly_representable_queries, dict(shift=0)),
    (qpins.test_verify_q8_equals_verify_for_exactly_representable_queries, dict(shift=3)),
]


@pytest.mark.parametrize("name", sorted(Q8_MUTANTS))
def test_q8_mutant_is_caught(name, monkeypatch):
    old, new = Q8_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.compile_oracle(path, os.path.join(tmp, f"lib{name}.so")))
        monkeypatch.setattr(qpins, "LIB", lib)
        caught = []
        for fn, kw in Q8_BATTERY:
            try:
                fn(**kw)
            except (AssertionError, oracle.OracleError):
                caught.append(fn.__name__)
        assert caught, f"no pin catches mutant {name}"
