"""Plant plausible mistakes in copies of the oracle; each must fail a pin.

Every mutant is a textual edit of hpc_oracle.c compiled into a temporary
library on the CPU. The pins of tests/_pins.py run against it in turn; the
mutant is caught when any of them raises. This shows the pins would notice a
dropped term, a wrong sign or index, or a transposed operand in the oracle.
"""
import os
import subprocess

import numpy as np
import pytest

import _pins as pins
import _pins_prologue as pp
import oracle

MUTANTS = {
    "no_softmax_scale": ("acc * scale", "acc"),
    "gqa_head_modulo": ("int h = qh / G;", "int h = qh % kv->Hkv;"),
    "floor_chunk_count": ("(len + OR_CHUNK_TOKENS - 1) / OR_CHUNK_TOKENS", "len / OR_CHUNK_TOKENS"),
    "batch_major_walk": (
        "    for (int h = 0; h < Hkv; ++h)\n        for (int b = 0; b < B; ++b)\n"
        "            for (long long c = 0; c < n[b]; ++c, ++g) {",
        "    for (int b = 0; b < B; ++b)\n        for (int h = 0; h < Hkv; ++h)\n"
        "            for (long long c = 0; c < n[b]; ++c, ++g) {"),
    "no_min_floor": ("if (bucket < m) bucket = m;", ""),
    "budget_rounds_down": ("long long bucket = (T + C - 1) / C;", "long long bucket = T / C;"),
    "combine_lse_unshifted": ("*lse = M + log(wsum);", "*lse = log(wsum);"),
    "e4m3_bias_8": ("e - 7);", "e - 8);"),
    "e4m3_subnormal_as_normal": ("ldexp((double)mant / 8.0, -6)", "ldexp(1.0 + (double)mant / 8.0, -7)"),
    "kv_head_major_layout": (
        "long long idx = ((page * OR_CHUNK_TOKENS + slot) * kv->Hkv + h) * OR_HEAD_DIM + dim;",
        "long long idx = ((page * kv->Hkv + h) * OR_CHUNK_TOKENS + slot) * OR_HEAD_DIM + dim;"),
    "scale_token_major": (
        "scale[(page * kv->Hkv + h) * OR_CHUNK_TOKENS + slot]",
        "scale[(page * OR_CHUNK_TOKENS + slot) * kv->Hkv + h]"),
    "softmax_sign": ("s[i] = exp(s[i] - mx);", "s[i] = exp(mx - s[i]);"),
    "partial_unnormalised": ("for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] /= sum;", ""),
    "lse_log2": ("*lse = mx + log(sum);", "*lse = mx + log2(sum);"),
    "tail_token_dropped": ("if (t1 > len) t1 = len;", "if (t1 > len) t1 = len - 1;"),
    "split_rank_off_by_one": ("t[5] = (int32_t)(i - split0[p]);", "t[5] = (int32_t)(i - split0[p] + 1);"),
    "combine_weights_unnormalised": ("for (int dd = 0; dd < OR_HEAD_DIM; ++dd) o[dd] /= wsum;", ""),
    "query_scale_dropped": ("qv[dd] = oracle_e4m3_to_f64(qrow[dd]) * qs;", "qv[dd] = oracle_e4m3_to_f64(qrow[dd]);"),
    "rope_sign": ("dst[i] = x[i] * c - x[i + half] * sn;", "dst[i] = x[i] * c + x[i + half] * sn;"),
    "rope_adjacent_pairs": ("dst[i + half] = x[i + half] * c + x[i] * sn;",
                            "dst[i + half] = x[i + half] * c + x[(i + 1) % half] * sn;"),
    "norm_without_eps": ("1.0 / sqrt(ss / OR_HEAD_DIM + eps)", "1.0 / sqrt(ss / OR_HEAD_DIM)"),
    "norm_weight_dropped": ("x[d] = x[d] * inv * (double)w[d];", "x[d] = x[d] * inv;"),
    "norm_sum_not_mean": ("1.0 / sqrt(ss / OR_HEAD_DIM + eps)", "1.0 / sqrt(ss + eps)"),
    "k_uses_q_weight": ("const float* w = j < Hq ? qw : kw;", "const float* w = qw;"),
    "causal_off_by_one": ("long long v = len - kv->q_len + qi + 1;", "long long v = len - kv->q_len + qi;"),
    "causal_reversed": ("long long v = len - kv->q_len + qi + 1;", "long long v = len - qi;"),
    "query_row_ignores_token": ("const long long row = ((long long)b * kv->q_len + qi) * kv->Hq + qh;",
                                "const long long row = (long long)b * kv->Hq + qh;"),
    "split_rows_token_major": ("long long row = ((long long)s * q_len + qi) * G + j;",
                               "long long row = ((long long)qi * plan[OR_H_TOTAL_SPLITS] + s) * G + j;"),
    "combine_reads_token_zero": ("long long srow = ((s0 + i) * q_len + qi) * G + j;",
                                 "long long srow = (s0 + i) * q_len * G + j;"),
}


def _all_pins():
    case_bf = pins.small_case([1, 63, 64, 65, 200, 333], hkv=2, hq=16, dtype="bf16", seed=11)
    case_f8 = pins.small_case([1, 65, 333], hkv=2, hq=16, dtype="fp8", seed=11)
    case_cb = pins.small_case([37, 128, 300, 1000, 0, 5], hkv=2, hq=16, seed=12)
    case_q8 = pins.small_case([1, 65, 333], hkv=2, hq=16, dtype="fp8", seed=15, q_dtype="fp8")
    case_mt = pins.small_case_mt([2, 65, 66, 200], 3, hkv=2, hq=16, seed=23)
    return [
        pins.check_e4m3_closed_forms,
        pins.check_golden_dynamic,
        pins.check_golden_static,
        lambda: pins.check_plan_random(trials=10),
        pins.check_attn_closed_forms,
        lambda: pins.check_attn_vs_sdpa(case_bf),
        lambda: pins.check_attn_vs_sdpa(case_f8),
        lambda: pins.check_attn_vs_sdpa(case_q8),
        lambda: pins.check_combine_equals_full(case_cb, 7, 2),
        pins.check_empty_request,
        lambda: pins.check_split_ranges(pins.small_case([37, 128, 300, 1000], seed=13), 16, 2),
        pins.check_e4m3_all_codes,
        pp.check_norm_at_position_zero,
        pp.check_rotation_keeps_pair_norms,
        pp.check_relative_position,
        lambda: pins.check_multitoken_vs_sdpa(case_mt),
        lambda: pins.check_multitoken_combine_equals_full(case_mt, 5, 1),
        pins.check_multitoken_short_requests,
        pins.check_plan_bruteforce_tiny,
    ]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(path), "-lm"],
                   check=True, capture_output=True)
    saved = oracle._load()
    oracle._lib = oracle.load_library(str(lib))
    caught = None
    try:
        for check in _all_pins():
            try:
                with np.errstate(all="ignore"):
                    check()
            except (AssertionError, ValueError, IndexError) as e:  # noqa: PERF203
                caught = e
                break
    finally:
        oracle._lib = saved
    assert caught is not None, f"mutant {name} passed every pin"
