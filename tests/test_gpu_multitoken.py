"""Several new tokens per request (speculative verification rows), CUDA path
against the float64 oracle through the C ABI (GPU only).

New token i of request b attends causally to tokens [0, L_b - q_len + i]. The
task map is the one-token map; every descriptor computes q_len x 8 rows. Same
bounds as the one-token path: BF16 KV max abs <= 2e-2 and mean abs <= 2e-3,
e4m3 KV max abs <= 6e-2, LSE <= 1e-3 abs.
"""
import numpy as np
import pytest
import torch

import _gpu
import oracle
from load_balanced_paged_02_gb300 import binding as hb
from load_balanced_paged_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# lengths around chunk edges, shorter than q_len, and empty
RAGGED = [1, 2, 5, 63, 64, 65, 66, 67, 70, 127, 128, 129, 130, 200, 333, 1000, 0, 4097]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hb.lib()


def case_for(lens, q_len, hkv=1, dtype="bf16", seed=0, pool=None):
    w = wl.Workload("t", len(lens), 8 * hkv, hkv, dtype, seed, lens=list(lens), pool_pages=pool,
                    q_len=q_len)
    return wl.make_case(w, device=DEV)


# (cache dtype, kernel): both kernels serve both cache dtypes
ENGINES = [("bf16", hb.ENGINE_MMA_SYNC), ("bf16", hb.ENGINE_TCGEN05), ("fp8", hb.ENGINE_MMA_SYNC),
           ("fp8", hb.ENGINE_TCGEN05)]
ENGINE_IDS = ["bf16-mma_sync", "bf16-tcgen05", "fp8-mma_sync", "fp8-tcgen05"]


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 5, 6, 7, 8])
def test_ragged_full(dtype, engine, q_len):
    case = case_for(RAGGED, q_len, hkv=2, dtype=dtype, seed=40 + q_len)
    if q_len == 1:
        case["q"] = case["q"].unsqueeze(1).contiguous()
    res = _gpu.run(case, num_ctas=152, min_chunks=2, engine=engine)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
def test_max_kv_heads(dtype, engine):
    """256 KV heads (the library's limit), 2048 query heads, three new tokens."""
    case = case_for([1, 100, 700, 0, 64], 3, hkv=256, dtype=dtype, seed=93)
    res = _gpu.run(case, num_ctas=152, min_chunks=2, engine=engine)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
@pytest.mark.parametrize("C,m", [(1, 0), (7, 1), (300, 4)])
def test_cta_budgets(dtype, engine, C, m):
    case = case_for(RAGGED, 6, hkv=1, dtype=dtype, seed=50 + C)
    res = _gpu.run(case, num_ctas=C, min_chunks=m, engine=engine)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
def test_static_split(dtype, engine):
    case = case_for([37, 128, 300, 1000, 0, 5, 4096], 4, hkv=2, dtype=dtype, seed=60)
    res = _gpu.run(case, static_splits=16, engine=engine)
    _gpu.check_plan_exact(res, case, static_splits=16)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("engine", [hb.ENGINE_MMA_SYNC, hb.ENGINE_TCGEN05], ids=["mma_sync", "tcgen05"])
def test_e4m3_peaky_scores_and_uneven_scales(engine):
    """e4m3 cache: a query aligned with one key (its score is 30, far above the
    first chunk's maximum, so the reference max moves) and K/V scales that vary
    by two orders of magnitude between tokens; the K scales weight the score
    columns and the V scales the value rows."""
    case = case_for([300, 700], 3, hkv=1, dtype="fp8", seed=65)
    g = torch.Generator(device="cpu").manual_seed(65)
    for cache, name in (("k_cache", "k_scale"), ("v_cache", "v_scale")):
        # codes / f and scale x f: the values keep their size (so the bf16
        # output rounding stays far below the bound) while the scales spread
        f = torch.exp(torch.empty(case[name].shape).uniform_(-2.3, 2.3, generator=g)).to(DEV)
        codes = case[cache].float() / f.permute(0, 2, 1).unsqueeze(-1)
        case[cache].copy_(codes.clamp(-448, 448).to(torch.float8_e4m3fn))
        case[name] *= f
    pt = case["page_table"].cpu().numpy()
    key = 290  # visible to new tokens 1 and 2 of request 0 (they see [0, 298] and [0, 299])
    pg, sl = int(pt[0, key // 64]), key % 64
    kv = case["k_cache"][pg, sl, 0].float() * case["k_scale"][pg, 0, sl]
    case["q"][0, :, 0] = (kv * (30.0 * 128 ** 0.5 / kv.dot(kv))).to(torch.bfloat16)
    res = _gpu.run(case, num_ctas=3, min_chunks=1, engine=engine)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_large_scores_move_the_reference_max(dtype):
    """Scores that grow along the sequence force the tcgen05 kernel to rescale
    its TMEM output several times (lazy rescale beyond 2^8); both kernels must
    still match the oracle."""
    case = case_for([700, 1500], 3, hkv=1, dtype=dtype, seed=66)
    pt = case["page_table"].cpu().numpy()
    for b, L in enumerate(case["seq_lens"].cpu().numpy()):
        for tok in range(0, int(L), 37):
            pg, sl = int(pt[b, tok // 64]), tok % 64
            if dtype == "fp8":  # e4m3 codes saturate: grow the token's K scale instead
                case["k_scale"][pg, 0, sl] *= 1 + tok / 300.0
            else:
                case["k_cache"][pg, sl, 0] = (case["k_cache"][pg, sl, 0].float() * (1 + tok / 300.0)).to(torch.bfloat16)
    case["q"] *= 2
    for engine in (hb.ENGINE_MMA_SYNC, hb.ENGINE_TCGEN05):
        res = _gpu.run(case, num_ctas=4, min_chunks=1, engine=engine)
        _gpu.check_full(case, res)


def test_one_token_through_the_multi_entry_matches_decode():
    """q_len = 1 through hpc_decode_attn_multi / hpc_decode_combine_multi gives
    the bytes of hpc_decode_attn / hpc_decode_combine."""
    case = case_for([37, 128, 300, 1000], 1, hkv=2, seed=61)
    ref = _gpu.run(case, num_ctas=16)
    q4 = case["q"].unsqueeze(1).contiguous()
    plan = ref["plan"]
    so, sl = hb.split_buffers(plan, q_len=1)
    L = hb.lib()
    rc = L.hpc_decode_attn_multi(
        hb._ptr(q4), 1, hb._ptr(case["k_cache"]), hb._ptr(case["v_cache"]), None, None, hb.KV_BF16,
        case["num_pages"], hb._ptr(case["page_table"]), case["page_table"].shape[1], hb._ptr(case["seq_lens"]),
        4, 16, 2, 128, 64, plan.ref(), hb._ptr(so), hb._ptr(sl), hb._stream(None))
    assert rc == 0
    out = torch.empty_like(q4)
    lse = torch.empty(q4.shape[:-1], dtype=torch.float32, device=DEV)
    hb.hpc_decode_combine(plan, so, sl, out, lse, 2)
    torch.cuda.synchronize()
    n = int(plan.buf[3].item())
    assert torch.equal(so[:n], ref["split_o"][:n]) and torch.equal(sl[:n], ref["split_lse"][:n])
    assert torch.equal(out[:, 0], ref["out"]) and torch.equal(lse[:, 0], ref["lse"])


def test_q_len_out_of_range_is_rejected():
    case = case_for([100, 200], 2, seed=62)
    plan = hb.hpc_decode_plan(case["seq_lens"], 1, 8, 2)
    so, sl = hb.split_buffers(plan, q_len=8)
    L = hb.lib()
    for bad in (0, -1, 9):
        rc = L.hpc_decode_attn_multi(
            hb._ptr(case["q"]), bad, hb._ptr(case["k_cache"]), hb._ptr(case["v_cache"]), None, None,
            hb.KV_BF16, case["num_pages"], hb._ptr(case["page_table"]), case["page_table"].shape[1],
            hb._ptr(case["seq_lens"]), 2, 8, 1, 128, 64, plan.ref(), hb._ptr(so), hb._ptr(sl),
            hb._stream(None))
        assert rc == 1, bad
        out = torch.empty((2, 8, 8, 128), dtype=torch.bfloat16, device=DEV)
        rc = L.hpc_decode_combine_multi(plan.ref(), bad, hb._ptr(so), hb._ptr(sl), hb._ptr(out), None, 2, 8, 1,
                                        128, hb._stream(None))
        assert rc == 1, bad
    assert hb.hpc_decode_read_error(plan) == 0


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
def test_invalid_page_id_sets_error_and_skips(dtype, engine):
    """A page id outside the pool sets the error bit and skips that chunk
    (nothing is loaded from it); the other request's rows are untouched."""
    case = case_for([200, 300], 3, hkv=1, dtype=dtype, seed=67)
    bad = case["page_table"].clone()
    bad[1, 2] = case["num_pages"] + 5
    res = _gpu.run(dict(case, page_table=bad), num_ctas=4, min_chunks=1, engine=engine)
    assert hb.hpc_decode_read_error(res["plan"]) & 4
    host = wl.to_numpy_case(case, requests=[0])
    rows = [(0, qi * 8 + h) for qi in range(3) for h in range(8)]
    ro, rl = oracle.attn_rows(host, rows)
    _gpu.assert_close(res["out"][0].float().cpu().numpy().reshape(-1, 128), res["lse"][0].cpu().numpy().reshape(-1),
                      ro, rl, case, "request 0")
    assert torch.isfinite(res["out"][1].float()).all()


@pytest.mark.parametrize("dtype,engine", ENGINES, ids=ENGINE_IDS)
def test_garbage_beyond_live_length_is_ignored(dtype, engine):
    """Slots past the live length of the last page hold NaN codes; the causal
    mask and the tail fill must keep them out of every row."""
    case = case_for([65, 130, 7, 200], 5, hkv=1, dtype=dtype, seed=63)
    pt = case["page_table"].cpu().numpy()
    for b, L in enumerate(case["seq_lens"].cpu().numpy()):
        if L % 64:
            pg = int(pt[b, (L - 1) // 64])
            for cache in (case["k_cache"], case["v_cache"]):
                if dtype == "fp8":
                    cache.view(torch.uint8)[pg, L % 64:] = 0x7F
                else:
                    cache[pg, L % 64:] = float("nan")
            if dtype == "fp8":
                case["k_scale"][pg, :, L % 64:] = float("nan")
                case["v_scale"][pg, :, L % 64:] = float("nan")
    res = _gpu.run(case, num_ctas=5, min_chunks=1, engine=engine)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("engine", [hb.ENGINE_MMA_SYNC, hb.ENGINE_TCGEN05], ids=["mma_sync", "tcgen05"])
def test_peaky_scores(engine):
    """A query aligned with one key: the row is dominated by that key, for the
    new token that sees it and not for the earlier ones."""
    case = case_for([300], 4, hkv=1, seed=64)
    pt = case["page_table"].cpu().numpy()
    key = 298  # visible to new tokens 2 and 3 (they see [0, 298] and [0, 299])
    k = case["k_cache"][int(pt[0, key // 64]), key % 64, 0].float()
    case["q"][0, :, 0] = (k * 4.0).to(torch.bfloat16)
    res = _gpu.run(case, num_ctas=3, min_chunks=1, engine=engine)
    _gpu.check_full(case, res)
    v = case["v_cache"][int(pt[0, key // 64]), key % 64, 0].float()
    out = res["out"][0, :, 0].float()
    assert torch.allclose(out[2], v, atol=0.05) and torch.allclose(out[3], v, atol=0.05)
    assert not torch.allclose(out[0], v, atol=0.05)


@pytest.mark.parametrize("name,q_len,engine", [("mixed", 2, None), ("mixed", 4, None), ("mixed", 6, None),
                                               ("mixed", 8, None), ("fp8", 6, hb.ENGINE_MMA_SYNC),
                                               ("fp8", 2, hb.ENGINE_TCGEN05), ("fp8", 8, hb.ENGINE_TCGEN05)])
def test_full_size_every_row(name, q_len, engine):
    """The full-size batch with q_len new tokens, in the launch configuration
    the benchmark times, against the oracle: on the bf16 batch every output
    row, LSE and split partial; on the e4m3 batch every row of every request
    and query head for new tokens 0 and q_len - 1 (the shortest and the
    longest causal limits; the float64 oracle takes ~17 s per new token
    there), plus the split/combine property over every row."""
    from dataclasses import replace
    w = replace(wl.WORKLOADS[name], q_len=q_len)
    case = wl.make_case(w, device=DEV)
    res = _gpu.run(case, num_ctas=hb.default_num_ctas(hb.kv_dtype_of(case["k_cache"])), min_chunks=w.min_chunks,
                   engine=engine)
    _gpu.check_plan_exact(res, case, min_chunks=w.min_chunks)
    if name == "mixed":
        _gpu.check_full(case, res, what=f"{name} q_len {q_len}")
    else:
        host = wl.to_numpy_case(case)
        B, Hq = w.batch, w.num_q_heads
        toks = sorted({0, q_len - 1})
        rows = [(b, qi * Hq + h) for b in range(B) for qi in toks for h in range(Hq)]
        ro, rl = oracle.attn_rows(host, rows)
        out = res["out"].float().cpu().numpy()[:, toks].reshape(-1, 128)
        lse = res["lse"].cpu().numpy()[:, toks].reshape(-1)
        _gpu.assert_close(out, lse, ro, rl, case, f"{name} q_len {q_len}, new tokens {toks}")
    _gpu.check_split_invariants(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0
