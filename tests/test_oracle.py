"""The float64 oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import _pins as pins

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def test_e4m3_decoder_all_codes():
    pins.check_e4m3_all_codes()


def test_e4m3_closed_forms():
    pins.check_e4m3_closed_forms()


def test_bf16_decoder():
    pins.check_bf16_codes()


def test_plan_golden_dynamic():
    pins.check_golden_dynamic()


def test_plan_golden_static():
    pins.check_golden_static()


def test_plan_bruteforce_tiny_grid():
    pins.check_plan_bruteforce_tiny()


def test_plan_invariants_random():
    pins.check_plan_random()


def test_static_plan_random():
    pins.check_static_random()


def test_plan_floor_prevents_over_partitioning():
    import oracle
    # 3 chunks over 100 CTAs: without the floor every chunk would get its own CTA
    p = oracle.parse_plan(oracle.plan([192], 1, 100, 2))
    assert p["header"]["bucket"] == 2 and p["header"]["used_ctas"] == 2
    assert [len(l) for l in p["lists"][:3]] == [1, 1, 0]
    # the floor never shrinks a large budget
    p = oracle.parse_plan(oracle.plan([64 * 1000], 1, 10, 2))
    assert p["header"]["bucket"] == 100


def test_plan_negative_length_sets_error_bit():
    import oracle
    p = oracle.parse_plan(oracle.plan([-5, 100], 1, 4, 1))
    assert p["header"]["error"] & 1
    assert p["header"]["total_chunks"] == 2


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_attn_matches_torch_sdpa(dtype):
    case = pins.small_case([1, 63, 64, 65, 200, 333], hkv=2, hq=16, dtype=dtype, seed=11)
    pins.check_attn_vs_sdpa(case)


def test_attn_with_e4m3_query_matches_torch_sdpa():
    """e4m3 Q with a scale per (request, query head), e4m3 KV."""
    case = pins.small_case([1, 63, 64, 65, 200, 333], hkv=2, hq=16, dtype="fp8", seed=15,
                           q_dtype="fp8")
    assert case["q"].dtype == np.uint8 and case["q_scale"].shape == (6, 16)
    pins.check_attn_vs_sdpa(case)


def test_combine_of_splits_with_e4m3_query():
    case = pins.small_case([37, 128, 300, 1000, 0, 5], hkv=2, hq=16, dtype="fp8", seed=16,
                           q_dtype="fp8")
    pins.check_combine_equals_full(case, 7, 2)


def test_attn_closed_forms():
    pins.check_attn_closed_forms()


def test_page_permutation_invariance():
    pins.check_page_permutation_invariance()


def test_empty_request():
    pins.check_empty_request()


@pytest.mark.parametrize("C,m", [(1, 0), (3, 1), (7, 2), (16, 2), (64, 3)])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_combine_of_splits_equals_unsplit(C, m, dtype):
    case = pins.small_case([37, 128, 300, 1000, 0, 5], hkv=2, hq=16, dtype=dtype, seed=12)
    pins.check_combine_equals_full(case, C, m)


def test_split_partials_are_plain_attention_over_their_range():
    case = pins.small_case([37, 128, 300, 1000], hkv=1, hq=8, seed=13)
    pins.check_split_ranges(case, 16, 2)


def test_single_chunk_is_plain_attention():
    # L <= 64: one chunk, one descriptor, the partial is the whole attention
    import oracle
    case = pins.small_case([50], seed=14)
    pb = oracle.plan(case["seq_lens"], 1, 8, 1)
    so, sl = oracle.attn_splits(pb, case)
    o, lse = oracle.attn_rows(case)
    assert so.shape[0] == 1
    assert np.array_equal(so[0], o) and np.array_equal(sl[0], lse)


# ------------------------------------------------------------------ several new tokens per request

@pytest.mark.parametrize("q_len", [2, 3, 6])
def test_multitoken_matches_masked_sdpa(q_len):
    case = pins.small_case_mt([1, 5, 63, 64, 65, 66, 130, 333], q_len, hkv=2, hq=16, seed=20 + q_len)
    pins.check_multitoken_vs_sdpa(case)


def test_multitoken_fp8_matches_masked_sdpa():
    case = pins.small_case_mt([3, 64, 65, 200], 4, hkv=1, hq=8, dtype="fp8", seed=30)
    pins.check_multitoken_vs_sdpa(case)


def test_multitoken_is_prefix_decode():
    case = pins.small_case_mt([6, 64, 65, 129, 1000], 6, hkv=2, hq=16, seed=31)
    pins.check_multitoken_is_prefix_decode(case)


@pytest.mark.parametrize("C,m", [(1, 0), (5, 1), (16, 2)])
@pytest.mark.parametrize("q_len", [2, 6])
def test_multitoken_combine_of_splits_equals_unsplit(C, m, q_len):
    case = pins.small_case_mt([37, 64, 65, 128, 129, 300, 1000, 0, 3], q_len, hkv=2, hq=16, seed=32)
    pins.check_multitoken_combine_equals_full(case, C, m)


def test_multitoken_split_ranges():
    case = pins.small_case_mt([65, 66, 128, 300], 3, hkv=1, hq=8, seed=33)
    pins.check_multitoken_split_ranges(case, 9, 1)


def test_multitoken_short_requests():
    pins.check_multitoken_short_requests()
