"""CUDA path against the float64 oracle, through the C ABI (GPU only).

Task maps must match byte for byte. Outputs: BF16 KV max abs <= 2e-2 and mean
abs <= 2e-3; e4m3 KV max abs <= 6e-2; LSE <= 1e-3 abs. Small cases compare
every output row and every split partial, and so do the full-size workloads
(tiny, uniform, mixed, skew, e4m3, e4m3 query, many short requests), for the
balanced map and for the static split-KV map of the same kernel.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hb.lib()


def case_for(lens, hkv=1, dtype="bf16", seed=0, pool=None, stride=None, q_dtype="bf16"):
    w = wl.Workload("t", len(lens), 8 * hkv, hkv, dtype, seed, lens=list(lens), pool_pages=pool,
                    q_dtype=q_dtype)
    return wl.make_case(w, device=DEV, stride=stride)


# ------------------------------------------------------------------ planner

@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_plan_bit_exact_workloads(name):
    w = wl.WORKLOADS[name]
    lens = torch.from_numpy(wl.draw_lengths(w).astype(np.int32)).to(DEV)
    C = w.num_ctas or hb.default_num_ctas(hb.KV_FP8_E4M3 if w.kv_dtype == "fp8" else hb.KV_BF16)
    plan = hb.hpc_decode_plan(lens, w.num_kv_heads, C, w.min_chunks)
    ref = oracle.plan(lens.cpu().numpy(), w.num_kv_heads, C, w.min_chunks)
    assert np.array_equal(plan.buf.cpu().numpy(), ref)
    st = hb.hpc_decode_plan_static(lens, w.num_kv_heads, w.static_splits)
    ref = oracle.plan_static(lens.cpu().numpy(), w.num_kv_heads, w.static_splits)
    assert np.array_equal(st.buf.cpu().numpy(), ref)


def test_plan_bit_exact_random_and_edges():
    rng = np.random.default_rng(123)
    cases = [([0], 1, 1, 0), ([0, 0, 0], 2, 5, 2), ([1], 1, 1, 0), ([64], 3, 7, 0),
             ([65, 1, 0, 4096], 8, 148, 2), ([10 ** 6], 8, 152, 2), ([37, 128, 300, 1000], 1, 16, 2)]
    for _ in range(60):
        B = int(rng.integers(1, 60))
        cases.append((rng.integers(0, 6000, size=B).tolist(), int(rng.integers(1, 9)),
                      int(rng.integers(1, 400)), int(rng.integers(0, 6))))
    # batch sizes and buckets at and next to powers of two: the planner divides by
    # both with a precomputed multiplier, whose shifts change at those points
    for B in (2, 3, 4, 5, 127, 128, 129, 1023, 1024, 1025):
        for C, m in ((1, 0), (B, 0), (3 * B + 1, 1), (256, 4)):
            cases.append((rng.integers(0, 5000, size=B).tolist(), int(rng.integers(1, 9)), C, m))
    # more than 1024 requests / pairs: several scan tiles, over several planner
    # blocks (one per 1024 pairs, at most 64)
    cases.append((rng.integers(0, 3000, size=3000).tolist(), 8, 304, 2))
    cases.append((rng.integers(0, 300, size=HB_MAX_B).tolist(), 1, 1000, 1))
    # 65 tiles: 64 blocks of two tiles each, the last 31 blocks without pairs
    cases.append((rng.integers(0, 400, size=8320).tolist(), 8, 152, 2))
    # 128 tiles, two per block, and a bucket well above one chunk
    cases.append((rng.integers(0, 200, size=HB_MAX_B).tolist(), 8, 1000, 2))
    # empty requests at block edges: pairs 1023 / 1024 / 2047 / 2048 have no chunks
    edge = rng.integers(1, 900, size=4096)
    edge[[1023, 1024, 2047, 2048, 4095]] = 0
    cases.append((edge.tolist(), 1, 152, 2))
    for lens, hkv, C, m in cases:
        sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
        plan = hb.hpc_decode_plan(sl, hkv, C, m)
        ref = oracle.plan(np.array(lens, dtype=np.int32), hkv, C, m)
        assert np.array_equal(plan.buf.cpu().numpy(), ref), (len(lens), hkv, C, m)
        S = int(rng.integers(1, 20))
        if hkv * len(lens) * S <= 1 << 20:
            st = hb.hpc_decode_plan_static(sl, hkv, S)
            assert np.array_equal(st.buf.cpu().numpy(), oracle.plan_static(np.array(lens, np.int32), hkv, S))


HB_MAX_B = 16384


def test_plan_negative_length_error_bit():
    sl = torch.tensor([-3, 100, 5], dtype=torch.int32, device=DEV)
    plan = hb.hpc_decode_plan(sl, 2, 4, 1)
    ref = oracle.plan(sl.cpu().numpy(), 2, 4, 1)
    assert np.array_equal(plan.buf.cpu().numpy(), ref)
    assert hb.hpc_decode_read_error(plan) & 1


# ------------------------------------------------------------------ attention, small (every row)

@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tiny_workload_full(dtype):
    w = wl.WORKLOADS["tiny"]
    case = case_for(w.lens, 1, dtype, seed=0, pool=64)
    res = _gpu.run(case, num_ctas=16, min_chunks=2)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("C,m", [(1, 0), (7, 1), (40, 2), (152, 2), (300, 4)])
def test_ragged_lengths_full(dtype, C, m):
    lens = [1, 63, 64, 65, 127, 200, 0, 333, 1000, 4097, 2, 640]
    case = case_for(lens, 2, dtype, seed=C + m)
    res = _gpu.run(case, num_ctas=C, min_chunks=m)
    _gpu.check_plan_exact(res, case, min_chunks=m)
    _gpu.check_full(case, res)
    out = res["out"].float().cpu().numpy()
    assert np.all(out[6] == 0) and np.all(np.isneginf(res["lse"][6].cpu().numpy()))


@pytest.mark.parametrize("C,m", [(1, 0), (7, 1), (152, 2), (300, 4)])
def test_e4m3_query_ragged_full(C, m):
    """e4m3 Q with per-(request, head) scales on the e4m3 cache: QK^T on e4m3
    operands, every row and every split against the oracle."""
    lens = [1, 63, 64, 65, 127, 200, 0, 333, 1000, 4097, 2, 640]
    case = case_for(lens, 2, "fp8", seed=C + m + 50, q_dtype="fp8")
    assert case["q"].dtype == torch.float8_e4m3fn
    res = _gpu.run(case, num_ctas=C, min_chunks=m)
    _gpu.check_plan_exact(res, case, min_chunks=m)
    _gpu.check_full(case, res)


def test_e4m3_query_static_and_peaky():
    lens = [37, 128, 300, 1000, 5000, 0, 64]
    case = case_for(lens, 2, "fp8", seed=57, q_dtype="fp8")
    res = _gpu.run(case, static_splits=4)
    _gpu.check_full(case, res)
    # a peaky query: scale x16 on one head of each request
    case["q_scale"][:, 3] *= 16.0
    res = _gpu.run(case, num_ctas=9)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("seed", [1, 2, 3, 4, 5])
def test_single_cta_many_descriptors(dtype, seed):
    """One or two CTAs drain every descriptor: the producer runs far ahead of
    the consumers, and short descriptors follow long ones, so the Q slots and
    the stage ring turn over while the previous contents are still in use."""
    lens = [1, 63, 64, 65, 127, 200, 0, 333, 1000, 4097, 2, 640, 1, 1, 70, 3]
    case = case_for(lens, 2, dtype, seed=seed)
    for C in (1, 2):
        res = _gpu.run(case, num_ctas=C, min_chunks=0)
        _gpu.check_plan_exact(res, case, min_chunks=0)
        _gpu.check_full(case, res)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_static_split_full(dtype):
    lens = [37, 128, 300, 1000, 5000, 0, 64]
    case = case_for(lens, 2, dtype, seed=5)
    res = _gpu.run(case, static_splits=4)
    _gpu.check_plan_exact(res, case, static_splits=4)
    _gpu.check_full(case, res)


@pytest.mark.parametrize("dtype,q_len,B,hkv", [
    ("bf16", 1, 400, 8), ("fp8", 1, 400, 8), ("bf16", 3, 140, 8),
    # more than two waves of the pair form; an odd q_len, whose consecutive
    # units change pair mid-warp-block; one KV head and an odd unit count
    ("bf16", 1, 700, 8), ("fp8", 1, 700, 8), ("bf16", 5, 130, 8), ("bf16", 1, 4865, 1)])
def test_many_short_requests_full(dtype, q_len, B, hkv):
    """Enough (KV-head pair, new token) tasks that the combine takes its
    one-warp-per-pair form (at least two blocks of 8 warps per SM on 152 SMs),
    with empty, one-chunk and multi-split pairs among them; every row and
    every split partial against the oracle."""
    rng = np.random.default_rng(80 + q_len + B)
    lens = rng.integers(0, 300, size=B)
    lens[::37] = 0
    lens[5] = 20000  # one request long enough to leave a multi-split pair
    w = wl.Workload("t", B, 8 * hkv, hkv, dtype, 81, lens=[int(x) for x in lens], q_len=q_len)
    case = wl.make_case(w, device=DEV)
    assert hkv * B * q_len >= 152 * 2 * 8
    res = _gpu.run(case, num_ctas=152, min_chunks=2)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_max_batch_full(dtype):
    """HPC_MAX_BATCH requests (short, ragged, every eleventh empty, one long)
    with one KV head: several scan tiles in the planner, ~15K descriptors over
    152 CTAs and the pair-form combine; every row and every split partial."""
    rng = np.random.default_rng(90)
    B = HB_MAX_B
    lens = rng.integers(0, 200, size=B)
    lens[::11] = 0
    lens[7] = 9000
    w = wl.Workload("t", B, 8, 1, dtype, 91, lens=[int(x) for x in lens])
    case = wl.make_case(w, device=DEV)
    res = _gpu.run(case, num_ctas=152, min_chunks=2)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("dtype,q_dtype", [("bf16", "bf16"), ("fp8", "bf16"), ("fp8", "fp8")])
def test_max_kv_heads_full(dtype, q_dtype):
    """HPC_MAX_KV_HEADS (256) KV heads, 2048 query heads: the KV tensor maps'
    head dimension and row stride at their largest, every row and split."""
    case = case_for([1, 100, 700, 0, 64], 256, dtype, seed=92, q_dtype=q_dtype)
    res = _gpu.run(case, num_ctas=152, min_chunks=2)
    _gpu.check_plan_exact(res, case, min_chunks=2)
    _gpu.check_full(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0


def test_suggested_cta_count():
    """One CTA per SM unless the busiest CTA of that plan holds at least 4
    descriptors and at least 0.15 per chunk of its budget; then the shallow
    instance's two per SM. Checked on the scope workloads and the Table 3
    mixes, whose measured step times the rule follows."""
    deep = hb.default_num_ctas(hb.KV_BF16)
    deep8 = hb.default_num_ctas(hb.KV_FP8_E4M3)
    shallow = 2 * hb.sm_count()
    for name, expect in (("tiny", deep), ("uniform", deep), ("mixed", deep), ("skew", deep), ("short", shallow)):
        w = wl.WORKLOADS[name]
        assert hb.suggest_num_ctas(wl.draw_lengths(w), w.num_kv_heads) == expect, name
    fp8 = wl.WORKLOADS["fp8"]
    assert hb.suggest_num_ctas(wl.draw_lengths(fp8), 8, hb.KV_FP8_E4M3) == deep8
    for mix, shape, expect in (("32x0.125K+32x4K", (64, 8), shallow), ("32x0.125K+32x4K", (8, 1), shallow),
                               ("64x0.5K", (64, 8), shallow), ("64x0.5K", (8, 1), deep8), ("64x4K", (64, 8), deep8),
                               ("1x128K+31x4K", (8, 1), deep8), ("2x32K+30x4K", (64, 8), deep8)):
        w = wl.table3_workload(mix, *shape)
        got = hb.suggest_num_ctas(wl.draw_lengths(w), w.num_kv_heads, hb.KV_FP8_E4M3)
        assert got == (2 * hb.sm_count() if expect == shallow else expect), (mix, shape)
    mix = wl.table3_workload("32x0.125K+32x4K", 64, 8)
    assert hb.suggest_num_ctas(wl.draw_lengths(mix), 8, q_len=2) == deep
    assert hb.suggest_num_ctas(np.zeros(5, np.int32), 8) == deep
    # the boundary: the first CTA (budget 68 chunks) holds the two-chunk requests
    # and the start of the first long one; 9 short requests make 10 descriptors
    # there (10 < 0.15 x 68), 10 make 11
    for n_short, expect in ((9, deep), (10, shallow)):
        lens = [128] * n_short + [64 * 64 * 40] * 4
        T = 2 * n_short + 4 * 64 * 40
        assert (T + deep - 1) // deep == 68
        assert hb.suggest_num_ctas(np.array(lens, np.int32), 1) == expect, n_short


@pytest.mark.parametrize("order", ["v_above_k", "k_above_v", "shared"])
def test_e4m3_scale_rows_in_one_copy_or_two(order):
    """The kernels fetch a page's two scale rows with one 3-D copy from the
    lower of the two arrays (K first when the K array is the lower, V first
    otherwise), and with two 2-D copies when both are one array (a caller
    sharing the scales of K and V). Each layout, every row and split against
    the oracle, on the one-token kernel and both multi-token kernels."""
    from dataclasses import replace
    lens = [1, 63, 64, 65, 127, 200, 0, 333, 1000, 4097]
    for q_len, engine in ((1, None), (2, hb.ENGINE_MMA_SYNC), (3, hb.ENGINE_TCGEN05)):
        w = wl.Workload("scales", len(lens), 16, 2, "fp8", 95 + q_len, lens=lens, q_len=q_len)
        case = wl.make_case(w, device=DEV)
        ks, vs = case["k_scale"], case["v_scale"]
        n = ks.numel()
        buf = torch.full((2 * n + 64,), float("nan"), dtype=torch.float32, device=DEV)
        lo, hi = buf[:n].view(ks.shape), buf[n + 64:].view(vs.shape)  # 256 bytes apart
        if order == "v_above_k":
            lo.copy_(ks)
            hi.copy_(vs)
            case = dict(case, k_scale=lo, v_scale=hi)
        elif order == "k_above_v":
            lo.copy_(vs)
            hi.copy_(ks)
            case = dict(case, k_scale=hi, v_scale=lo)
        else:
            lo.copy_(ks)
            case = dict(case, k_scale=lo, v_scale=lo)
        for C in (7, 40):
            res = _gpu.run(case, num_ctas=C, min_chunks=1, engine=engine)
            _gpu.check_plan_exact(res, case, min_chunks=1)
            _gpu.check_full(case, res, what=f"{order} q_len {q_len} C={C}")
            assert hb.hpc_decode_read_error(res["plan"]) == 0


@pytest.mark.parametrize("q_len", [1, 2])
def test_combine_rows_with_hundreds_of_partials(q_len):
    """A request split into 300 partials (600 chunks on a map for 600 CTAs):
    the row combine of small grids keeps the first 128 LSEs of a row in
    registers and walks its partials in tiles of 256, sixteen at a time; every
    row and split against the oracle."""
    lens = [38400, 5000, 1, 0]
    w = wl.Workload("longpair", len(lens), 8, 1, "bf16", 96 + q_len, lens=lens, q_len=q_len)
    case = wl.make_case(w, device=DEV)
    res = _gpu.run(case, num_ctas=600, min_chunks=1)
    _gpu.check_plan_exact(res, case, min_chunks=1)
    parsed = oracle.parse_plan(res["plan"].buf.cpu().numpy())
    assert int(parsed["pair_nsplit"].max()) == 300
    _gpu.check_full(case, res, what=f"300 partials, q_len {q_len}")


def test_all_lengths_zero():
    case = case_for([0, 0, 0], 1, seed=6, pool=4)
    res = _gpu.run(case, num_ctas=8)
    assert np.all(res["out"].float().cpu().numpy() == 0)
    assert np.all(np.isneginf(res["lse"].cpu().numpy()))


def test_plan_reused_across_layers():
    """One task map per step serves every layer (different caches, same lengths)."""
    lens = [100, 3000, 64, 777]
    a = case_for(lens, 2, seed=7)
    b = case_for(lens, 2, seed=8)
    b["page_table"], b["seq_lens"] = a["page_table"], a["seq_lens"]
    res_a = _gpu.run(a, num_ctas=20)
    res_b = _gpu.run(b, plan=res_a["plan"])
    _gpu.check_full(a, res_a)
    _gpu.check_full(b, res_b)


def test_peaky_scores():
    """Q scaled x8 with a planted key equal to q: the softmax is far from flat,
    so max tracking and rescaling matter. Checked also by relative norm."""
    lens = [3000, 130, 64 * 9 + 5]
    case = case_for(lens, 1, seed=9)
    q = case["q"].float() * 8.0
    case["q"] = q.to(torch.bfloat16)
    pt = case["page_table"].cpu().numpy()
    for b, L in enumerate(lens):
        t = (b * 977) % L
        case["k_cache"][pt[b, t // 64], t % 64, 0] = case["q"][b, 0] / 8.0
    res = _gpu.run(case, num_ctas=9)
    _gpu.check_full(case, res)
    host = wl.to_numpy_case(case)
    ro, _ = oracle.attn_rows(host)
    got = res["out"].float().cpu().numpy().reshape(-1, 128)
    rel = np.linalg.norm(got - ro, axis=1) / np.maximum(np.linalg.norm(ro, axis=1), 1e-30)
    assert rel.max() < 1e-2


def test_invalid_page_id_sets_error_and_skips():
    lens = [200, 300]
    case = case_for(lens, 1, seed=10)
    bad = case["page_table"].clone()
    bad[1, 2] = case["num_pages"] + 5
    case_bad = dict(case, page_table=bad)
    res = _gpu.run(case_bad, num_ctas=4)
    assert hb.hpc_decode_read_error(res["plan"]) & 4
    # request 0 is untouched by the bad page of request 1
    host = wl.to_numpy_case(case)
    ro, rl = oracle.attn_rows(host, [(0, h) for h in range(8)])
    _gpu.assert_close(res["out"][0].float().cpu().numpy(), res["lse"][0].cpu().numpy(), ro, rl, case)


def test_garbage_beyond_live_length_is_ignored():
    """NaN bits in the unused slots of a request's last page must not leak."""
    lens = [70, 129]
    case = case_for(lens, 1, seed=11)
    pt = case["page_table"].cpu().numpy()
    for b, L in enumerate(lens):
        last = pt[b, (L - 1) // 64]
        case["k_cache"][last, L % 64:] = float("nan")
        case["v_cache"][last, L % 64:] = float("nan")
    res = _gpu.run(case, num_ctas=3)
    _gpu.check_full(case, res, check_splits=False)


def test_garbage_beyond_live_length_is_ignored_fp8():
    lens = [70, 129]
    case = case_for(lens, 1, "fp8", seed=12)
    pt = case["page_table"].cpu().numpy()
    for b, L in enumerate(lens):
        last = pt[b, (L - 1) // 64]
        case["k_cache"].view(torch.uint8)[last, L % 64:] = 0x7F
        case["v_cache"].view(torch.uint8)[last, L % 64:] = 0x7F
        case["k_scale"][last, :, L % 64:] = float("inf")
        case["v_scale"][last, :, L % 64:] = float("nan")
    res = _gpu.run(case, num_ctas=3)
    _gpu.check_full(case, res, check_splits=False)


def test_step_host_matches_device_path():
    lens = [500, 64, 1300, 7]
    case = case_for(lens, 2, seed=13)
    res = _gpu.run(case, num_ctas=10)
    B, Hq, D = case["q"].shape
    ws_bytes = hb.step_workspace_bytes(B, Hq, 2, case["page_table"].shape[1], 10)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    h_q = case["q"].cpu().pin_memory()
    h_sl = case["seq_lens"].cpu().pin_memory()
    h_pt = case["page_table"].cpu().pin_memory()
    h_out = torch.empty_like(h_q).pin_memory()
    h_lse = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    hb.hpc_decode_step_host(h_q, h_sl, h_pt, case["k_cache"], case["v_cache"], ws, h_out, h_lse,
                            num_ctas=10, num_pages=case["num_pages"])
    torch.cuda.synchronize()
    assert torch.equal(h_out, res["out"].cpu())
    assert torch.equal(h_lse, res["lse"].cpu())


def test_step_host_pageable_buffers_take_the_copy_path():
    """Pageable host buffers go through cudaMemcpyAsync (the mapped ones
    through the staging kernel and the combine): same bytes either way."""
    lens = [500, 64, 1300, 7]
    case = case_for(lens, 2, seed=14)
    res = _gpu.run(case, num_ctas=10)
    B, Hq, D = case["q"].shape
    ws = torch.empty(hb.step_workspace_bytes(B, Hq, 2, case["page_table"].shape[1], 10), dtype=torch.uint8,
                     device=DEV)
    for pinned in (False, True):
        h = [case[k].cpu() for k in ("q", "seq_lens", "page_table")]
        h_out = torch.full_like(h[0], float("nan"))
        h_lse = torch.full((B, Hq), float("nan"), dtype=torch.float32)
        if pinned:
            h = [t.pin_memory() for t in h]
            h_out, h_lse = h_out.pin_memory(), h_lse.pin_memory()
        hb.hpc_decode_step_host(h[0], h[1], h[2], case["k_cache"], case["v_cache"], ws, h_out, h_lse,
                                num_ctas=10, num_pages=case["num_pages"])
        torch.cuda.synchronize()
        assert torch.equal(h_out, res["out"].cpu()), f"pinned={pinned}"
        assert torch.equal(h_lse, res["lse"].cpu()), f"pinned={pinned}"


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_step_graph_matches_step_host(dtype):
    """The captured step (hpc_decode_step_graph_*) gives the bytes of
    hpc_decode_step_host, and picks up new inputs written in place into its
    pinned host buffers (new query, new lengths, so a new task map)."""
    lens = [500, 64, 1300, 7, 0, 65]
    case = case_for(lens, 2, dtype=dtype, seed=17)
    B, Hq, D = case["q"].shape
    C = 12
    ws_bytes = hb.step_workspace_bytes(B, Hq, 2, case["page_table"].shape[1], C)
    ws_a = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    ws_b = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    h_q = case["q"].cpu().pin_memory()
    h_sl = case["seq_lens"].cpu().pin_memory()
    h_pt = case["page_table"].cpu().pin_memory()
    outs = [torch.empty_like(h_q).pin_memory() for _ in range(2)]
    lses = [torch.empty((B, Hq), dtype=torch.float32).pin_memory() for _ in range(2)]
    kw = dict(k_scale=case["k_scale"], v_scale=case["v_scale"], num_ctas=C, num_pages=case["num_pages"])
    g = hb.StepGraph(h_q, h_sl, h_pt, case["k_cache"], case["v_cache"], ws_b, outs[1], lses[1], **kw)
    try:
        for step in range(3):
            if step > 0:  # new inputs, in place
                h_q.copy_(torch.randn(h_q.shape, generator=torch.Generator().manual_seed(step)).to(h_q.dtype))
                # (each new length within the request's pages)
                h_sl.copy_(torch.tensor([500 - 150 * step, 64 - step, 1300 - 200 * step, 7 - 2 * step, 0,
                                         65 - 30 * step], dtype=torch.int32))
            outs[1].fill_(float("nan"))
            hb.hpc_decode_step_host(h_q, h_sl, h_pt, case["k_cache"], case["v_cache"], ws_a, outs[0], lses[0],
                                    **kw)
            g.launch()
            torch.cuda.synchronize()
            assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), f"step {step}"
            assert torch.equal(lses[0].view(torch.int32), lses[1].view(torch.int32)), f"step {step}"
        # and the last step against the oracle
        host = wl.to_numpy_case(dict(case, q=h_q.to(DEV), seq_lens=h_sl.to(DEV)))
        ro, rl = oracle.attn_rows(host)
        _gpu.assert_close(outs[1].float().numpy(), lses[1].numpy(), ro.reshape(B, Hq, 128), rl.reshape(B, Hq),
                          case, "captured step")
    finally:
        g.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_cuda_graph_replay_recomputes_from_device_inputs(dtype):
    """The step (plan -> attn -> combine, chained with programmatic dependent
    launch) captures into one CUDA graph; each replay re-plans from the lengths
    in device memory, so new lengths and new Q give new, correct outputs."""
    lens_a = [100, 3000, 64, 777, 0]
    lens_b = [2000, 5, 640, 3100, 129]
    cap = [max(x, y) for x, y in zip(lens_a, lens_b)]
    case = case_for(cap, 2, dtype, seed=21)
    Hkv = 2
    case["seq_lens"].copy_(torch.tensor(lens_a, dtype=torch.int32))
    plan = hb.hpc_decode_plan(case["seq_lens"], Hkv, 24, 2)
    so, sl = hb.split_buffers(plan)
    out = torch.empty_like(case["q"])
    lse = torch.empty(case["q"].shape[:2], dtype=torch.float32, device=DEV)

    def step():
        hb.hpc_decode_plan(case["seq_lens"], Hkv, 24, 2, plan=plan)
        hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                           case["seq_lens"], plan, so, sl, case["k_scale"], case["v_scale"],
                           num_pages=case["num_pages"])
        hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    gen = torch.Generator(device=DEV)
    gen.manual_seed(5)
    for lens in (lens_a, lens_b, lens_a):
        case["seq_lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        case["q"].copy_(torch.randn(case["q"].shape, generator=gen, device=DEV).to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        res = dict(plan=plan, split_o=so, split_lse=sl, out=out, lse=lse)
        _gpu.check_plan_exact(res, case, min_chunks=2)
        _gpu.check_full(case, res)


def test_many_steps_chained_without_sync():
    """Back-to-back steps on one stream with no host synchronisation between
    them: each kernel waits for its predecessor's output before reading it."""
    lens = [1000, 64, 4097, 300]
    case = case_for(lens, 2, seed=22)
    plan = hb.hpc_decode_plan(case["seq_lens"], 2, 16, 2)
    so, sl = hb.split_buffers(plan)
    outs = []
    for k in range(6):
        hb.hpc_decode_plan(case["seq_lens"], 2, 16, 2, plan=plan)
        hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                           case["seq_lens"], plan, so, sl, num_pages=case["num_pages"])
        o = torch.empty_like(case["q"])
        l = torch.empty(case["q"].shape[:2], dtype=torch.float32, device=DEV)
        hb.hpc_decode_combine(plan, so, sl, o, l, 2)
        outs.append((o, l))
    torch.cuda.synchronize()
    res = dict(plan=plan, split_o=so, split_lse=sl, out=outs[-1][0], lse=outs[-1][1])
    _gpu.check_full(case, res)
    for o, l in outs:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


# ------------------------------------------------------------------ full-size workloads

def test_uniform_workload_full():
    w = wl.WORKLOADS["uniform"]
    case = wl.make_case(w, device=DEV)
    res = _gpu.run(case, num_ctas=w.num_ctas, min_chunks=w.min_chunks)
    _gpu.check_plan_exact(res, case, min_chunks=w.min_chunks)
    _gpu.check_full(case, res, check_splits=True, what="uniform")
    _gpu.check_split_invariants(case, res)


@pytest.mark.parametrize("name", ["mixed", "skew", "fp8", "fp8q", "short"])
def test_full_size_workload_every_row(name):
    """The full batch in the launch configuration the benchmark times: every
    output row and LSE and every split partial of the balanced map against the
    float64 oracle; then the static split-KV schedule of the same kernel
    (S = 16), again every row (and every split partial on the bf16 batches)."""
    w = wl.WORKLOADS[name]
    case = wl.make_case(w, device=DEV)
    host = wl.to_numpy_case(case)
    rows = oracle.attn_rows(host)
    # the CTA count the library suggests for the batch (one per SM; two per SM,
    # the shallow instance, for the batch of many short requests)
    C = hb.suggest_num_ctas(case["seq_lens"], w.num_kv_heads, hb.kv_dtype_of(case["k_cache"]), w.min_chunks)
    res = _gpu.run(case, num_ctas=C, min_chunks=w.min_chunks)
    _gpu.check_plan_exact(res, case, min_chunks=w.min_chunks)
    _gpu.check_full(case, res, host=host, rows=rows, what=f"{name} balanced (C={C})")
    _gpu.check_split_invariants(case, res)
    assert hb.hpc_decode_read_error(res["plan"]) == 0
    del res
    st = _gpu.run(case, static_splits=w.static_splits)
    _gpu.check_plan_exact(st, case, static_splits=w.static_splits)
    # (the e4m3 batches' static partials, 7824 of them, are left to the
    # split/combine property: the oracle takes ~17 s per pass over that batch)
    _gpu.check_full(case, st, host=host, rows=rows, check_splits=w.kv_dtype != "fp8",
                    what=f"{name} static (S={w.static_splits})")
    _gpu.check_split_invariants(case, st)
