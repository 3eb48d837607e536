"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a one-line edit of oracle/pgqa_oracle.c (a dropped term, a
wrong sign or index, a swapped operand), compiled into a temporary library on
the CPU.  If a mutant passed every pin, the pins would not be strong enough to
trust the oracle against that kind of mistake.
"""
import numpy as np
import pytest

import oracle
import oracle_pins

MUTANTS = {
    "kv_head_modulo": ("const int kvh = h / g;\n    const int d = p->d;",
                       "const int kvh = h % p->Hkv;\n    const int d = p->d;"),
    "no_max_shift_in_lse": ("*lse = m + log(z);\n    free(w);", "*lse = log(z);\n    free(w);"),
    "missing_normalisation": ("o[c] = acc / z;", "o[c] = acc;"),
    "values_from_keys": ("acc += w[j - j0] * V[j * d + c];", "acc += w[j - j0] * K[j * d + c];"),
    "page_ignores_indptr": ("int64_t page = kv_indices[kv_indptr[b] + j / page_size];",
                            "int64_t page = kv_indices[j / page_size];"),
    "offset_not_modulo": ("int64_t off = j % page_size;", "int64_t off = (j + 1) % page_size;"),
    "causal_off_by_one": ("allowed = n - L + i + 1;\n            if (allowed < 0) allowed = 0;\n"
                          "            if (allowed > n) allowed = n;\n        }\n        for",
                          "allowed = n - L + i;\n            if (allowed < 0) allowed = 0;\n"
                          "            if (allowed > n) allowed = n;\n        }\n        for"),
    "causal_top_left": ("allowed = n - L + i + 1;\n            if (allowed < 0) allowed = 0;\n"
                        "            if (allowed > n) allowed = n;\n        }\n        for",
                        "allowed = i + 1;\n            if (allowed < 0) allowed = 0;\n"
                        "            if (allowed > n) allowed = n;\n        }\n        for"),
    "merge_unnormalised": ("double w = exp(lse_parts[s] - m) / z;", "double w = exp(lse_parts[s] - m);"),
    "merge_lse_drops_max": ("*lse = m + log(z);\n}", "*lse = log(z);\n}"),
    "scale_one_over_d": ("scale = 1.0 / sqrt((double)d);\n    problem_t",
                         "scale = 1.0 / (double)d;\n    problem_t"),
    "kv_len_whole_pages": ("return (npages - 1) * page_size + last_page_len[b];",
                           "return (npages - 1) * page_size + last_page_len[b] - 1;"),
    "fp16_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "bf16_shift": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "append_v_from_k": ("memcpy(v_pool + s * row_bytes, v + t * row_bytes",
                        "memcpy(v_pool + s * row_bytes, k + t * row_bytes"),
    "softmax_sign": ("w[j - j0] = exp(w[j - j0] - m);", "w[j - j0] = exp(m - w[j - j0]);"),
    "query_head_index": ("qv[c] = oracle_widen(p->q[(r * p->Hq + h) * (int64_t)d + c], p->dtype);",
                         "qv[c] = oracle_widen(p->q[(r * p->Hq + (h / g) * g) * (int64_t)d + c], p->dtype);"),
    "narrow_via_binary32": ("double a = fabs(x);\n    if (a == 0.0)", "double a = fabs((double)(float)x);\n    if (a == 0.0)"),
    "narrow_ties_away": ("(frac == 0.5 && fmod(fl, 2.0) != 0.0)", "(frac == 0.5)"),
    "narrow_no_subnormal_floor": ("if (e < emin)\n        e = emin;", "if (e < emin - 64)\n        e = emin;"),
    "narrow_truncates": ("if (frac > 0.5 || (frac", "if (frac > 1.5 || (frac"),
    "rope_turns_backwards": ("const double c = cos(phi), s = sin(phi);", "const double c = cos(phi), s = -sin(phi);"),
    "rope_freq_exponent": ("pow(theta, -2.0 * i / d)", "pow(theta, -1.0 * i / d)"),
    "rope_adjacent_pairs": ("const double a = x[base + i], b = x[base + i + half];",
                            "const double a = x[base + i], b = x[base + (i + half + 1) % d];"),
    "rope_second_sign": ("y[base + i + half] = b * c + a * s;", "y[base + i + half] = b * c - a * s;"),
    "rope_first_position": ("const double pos = (double)positions[r];", "const double pos = (double)positions[0];"),
    # more attention, merge and decoding mistakes
    "causal_global_row": ("int64_t i = r - r0;\n        int64_t allowed = n;", "int64_t i = r;\n        int64_t allowed = n;"),
    "kv_len_full_last_page": ("return (npages - 1) * page_size + last_page_len[b];", "return npages * page_size;"),
    "gather_first_kv_head": ("int64_t base = ((page * page_size + off) * Hkv + kvh) * (int64_t)d;",
                             "int64_t base = ((page * page_size + off) * Hkv + 0) * (int64_t)d;"),
    "merge_uniform_weights": ("double w = exp(lse_parts[s] - m) / z;", "double w = 1.0 / n;"),
    "fp16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    # page-table checks, the append's skip rule, empty slices and the merge loop
    "page_check_pool_end": ("kv_indices[i] >= num_pages)", "kv_indices[i] > num_pages)"),
    "page_check_negative_index": ("if (kv_indices[i] < 0 || kv_indices[i]", "if (kv_indices[i]"),
    "page_check_empty_len": ("if (npages == 0 && last_page_len[b] != 0)", "if (npages == 0 && last_page_len[b] < 0)"),
    "append_skips_slot_zero": ("if (s < 0)\n            continue;", "if (s <= 0)\n            continue;"),
    "empty_range_lse_zero": ("*lse = -INFINITY;\n        return ORACLE_OK;", "*lse = 0.0;\n        return ORACLE_OK;"),
    "merge_skips_first": ("for (int s = 0; s < n; ++s) {\n        if (lse_parts[s] == -INFINITY)",
                          "for (int s = 1; s < n; ++s) {\n        if (lse_parts[s] == -INFINITY)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.build(mutated, tmp_path / "libmutant.so", force=True))
    caught = []
    for pin_name, pin in sorted(oracle_pins.PINS.items()):
        try:
            with np.errstate(invalid="ignore", over="ignore", divide="ignore"):  # a mutant may yield NaN/inf
                pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin_name)
    assert caught, f"mutant {name} passed every pin"
