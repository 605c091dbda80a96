"""Checks that pin the float64 oracle to facts fixed outside the oracle.

Each check raises AssertionError when the oracle disagrees. They are used by
tests/test_oracle.py (on the oracle as built) and tests/test_oracle_mutants.py
(on copies of the oracle with a planted mistake, which must fail at least one
check). Sources: the HPC-Ops/SGLang blog ("Scheduling around live KV work")
and the vLLM x HPC-Ops blog ("解决方案：按步负载均衡的 decode 调度器").
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

import oracle
from load_balanced_paged_02_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ numbers

def check_e4m3_all_codes():
    """All 256 e4m3fn codes against torch's float8_e4m3fn -> float64 (a library decode)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)), "NaN codes differ"
    assert np.array_equal(ref[~nan], got[~nan]), "finite e4m3 values differ"


def check_e4m3_closed_forms():
    """Values fixed by the OCP FP8 definition."""
    assert oracle.e4m3_to_f64(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0xB8) == -1.0
    assert oracle.e4m3_to_f64(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert math.isnan(oracle.e4m3_to_f64(0x7F)) and math.isnan(oracle.e4m3_to_f64(0xFF))


def check_bf16_codes():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# ------------------------------------------------------------------ planner

def read_golden(name):
    params, header, descs = None, None, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "params":
                params = [[int(x) for x in rest[0].split(",")]] + [int(x) for x in rest[1:]]
            elif key == "header":
                header = [int(x) for x in rest]
            elif key == "desc":
                descs.append(tuple(int(x) for x in rest))
    return params, header, descs


def plan_descs(parsed):
    """Flatten per-CTA lists into (cta, h, b, c0, c1, split, rank, nsplit) tuples."""
    out = []
    for j, lst in enumerate(parsed["lists"]):
        for t in lst:
            out.append((j,) + t[:7])
    return out


def check_golden_dynamic():
    (lens, hkv, C, m), header, descs = read_golden("plan_tiny_dynamic.txt")
    p = oracle.parse_plan(oracle.plan(lens, hkv, C, m))
    h = p["header"]
    assert [h["total_chunks"], h["bucket"], h["used_ctas"], h["total_splits"]] == header
    assert plan_descs(p) == descs
    assert [len(l) for l in p["lists"][12:]] == [0, 0, 0, 0]


def check_golden_static():
    (lens, hkv, S), header, descs = read_golden("plan_tiny_static4.txt")
    p = oracle.parse_plan(oracle.plan_static(lens, hkv, S))
    h = p["header"]
    assert [h["total_chunks"], h["bucket"], h["used_ctas"], h["total_splits"]] == header
    assert plan_descs(p) == descs


def naive_plan(lens, hkv, C, m):
    """Second, deliberately naive formulation: label every chunk with its bucket,
    then group equal (pair, bucket) labels. Returns per-CTA descriptor lists."""
    n = [max(0, -(-int(L) // 64)) if L > 0 else 0 for L in lens]
    chunks = [(h, b, c) for h in range(hkv) for b in range(len(lens)) for c in range(n[b])]
    T = len(chunks)
    bucket = max(-(-T // C), m, 1)
    groups = {}
    order = []
    for g, (h, b, c) in enumerate(chunks):
        key = (g // bucket, h, b)
        if key not in groups:
            groups[key] = [c, c + 1]
            order.append(key)
        else:
            groups[key][1] = c + 1
    lists = [[] for _ in range(C)]
    for s, key in enumerate(order):
        lists[key[0]].append((key[1], key[2], groups[key][0], groups[key][1], s))
    return lists, bucket, T


def check_plan_against_naive(lens, hkv, C, m):
    p = oracle.parse_plan(oracle.plan(lens, hkv, C, m))
    lists, bucket, T = naive_plan(lens, hkv, C, m)
    got = [[t[:5] for t in lst] for lst in p["lists"]]
    assert got == lists, (lens, hkv, C, m)
    assert p["header"]["bucket"] == bucket and p["header"]["total_chunks"] == T


def check_plan_invariants(parsed, lens, hkv, m=None, static_splits=None):
    """Properties any correct task map has, whatever the formulation."""
    h = parsed["header"]
    B, C = len(lens), h["num_ctas"]
    n = [(-(-int(L) // 64)) if L > 0 else 0 for L in lens]
    cover = {}
    prev_key = None
    split = 0
    for j, lst in enumerate(parsed["lists"]):
        load = 0
        for t in lst:
            kh, b, c0, c1, s, rank, ns = t[:7]
            assert 0 <= kh < hkv and 0 <= b < B and 0 <= c0 < c1 <= n[b]
            assert s == split, "split indices follow walk order"
            split += 1
            key = (kh, b, c0)
            assert prev_key is None or key > prev_key, "walk is head-major, request, chunk"
            prev_key = key
            for c in range(c0, c1):
                assert (kh, b, c) not in cover, "chunk assigned twice"
                cover[(kh, b, c)] = j
            load += c1 - c0
        if static_splits is None:
            assert load <= h["bucket"], "bucket over budget"
            if 0 < j + 1 < h["used_ctas"]:
                assert load == h["bucket"], "every used CTA but the last is full"
        else:
            assert len(lst) <= 1
    assert len(cover) == hkv * sum(n), "every chunk assigned exactly once"
    assert split == h["total_splits"]
    if static_splits is None:
        T = hkv * sum(n)
        assert h["bucket"] == max(-(-T // C), m, 1)
        assert h["bucket"] >= m, "minimum per-CTA work respected"
        assert h["used_ctas"] == (-(-T // h["bucket"]) if T else 0)
        # a descriptor is a maximal run: consecutive descriptors of one pair sit in different CTAs
    nsplit, split0 = parsed["pair_nsplit"], parsed["pair_split0"]
    assert int(nsplit.sum()) == split
    for p in range(hkv * B):
        kh, b = divmod(p, B)
        ds = [t for lst in parsed["lists"] for t in lst if t[0] == kh and t[1] == b]
        assert len(ds) == nsplit[p]
        if ds:
            assert ds[0][4] == split0[p]
            assert [d[5] for d in ds] == list(range(len(ds)))
            assert all(d[6] == len(ds) for d in ds)
            assert ds[0][2] == 0 and ds[-1][3] == n[b]
            for a, bb in zip(ds, ds[1:]):
                assert a[3] == bb[2], "splits of a pair are contiguous"


def check_plan_bruteforce_tiny():
    """Every input on a small grid (B <= 3, L <= 200, Hkv <= 2, C <= 6, m <= 3)."""
    Ls = [0, 1, 64, 65, 128, 200]
    count = 0
    for B in (1, 2, 3):
        for lens in itertools.product(Ls, repeat=B):
            for hkv in (1, 2):
                for C in range(1, 7):
                    for m in range(0, 4):
                        check_plan_against_naive(list(lens), hkv, C, m)
                        count += 1
    assert count > 1000


def check_plan_random(seed=0, trials=40):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 5000, size=B).tolist()
        hkv = int(rng.integers(1, 9))
        C = int(rng.integers(1, 200))
        m = int(rng.integers(0, 6))
        buf = oracle.plan(lens, hkv, C, m)
        parsed = oracle.parse_plan(buf)
        check_plan_invariants(parsed, lens, hkv, m=m)
        check_plan_against_naive(lens, hkv, C, m)


def check_static_random(seed=1, trials=30):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        B = int(rng.integers(1, 12))
        lens = rng.integers(0, 3000, size=B).tolist()
        hkv = int(rng.integers(1, 4))
        S = int(rng.integers(1, 20))
        parsed = oracle.parse_plan(oracle.plan_static(lens, hkv, S))
        check_plan_invariants(parsed, lens, hkv, static_splits=S)
        n = [(-(-L // 64)) if L > 0 else 0 for L in lens]
        for j, lst in enumerate(parsed["lists"]):
            pair, s = divmod(j, S)
            kh, b = divmod(pair, B)
            q = -(-n[b] // S)
            if q and s * q < n[b]:
                assert lst and lst[0][:4] == (kh, b, s * q, min((s + 1) * q, n[b]))
            else:
                assert not lst


# ------------------------------------------------------------------ attention

def small_case(lens, hkv=1, hq=8, dtype="bf16", seed=0, pool=None, q_dtype="bf16"):
    w = wl.Workload("pin", len(lens), hq, hkv, dtype, seed, lens=list(lens), pool_pages=pool,
                    q_dtype=q_dtype)
    case = wl.make_case(w, device="cpu")
    return wl.to_numpy_case(case)


def dense_kv(case, b, kv_head):
    """Gather request b's K/V of one KV head as float64 through its page table,
    decoding with torch's own bf16 / float8_e4m3fn conversions."""
    L = int(case["seq_lens"][b])
    pages = case["page_table"][b]

    def dec(cache, scale):
        t = torch.from_numpy(cache)
        if cache.dtype == np.uint8:
            x = t.view(torch.float8_e4m3fn).to(torch.float64)
        else:
            x = t.view(torch.int16).view(torch.bfloat16).to(torch.float64)
        rows = []
        for tok in range(L):
            pg, sl = pages[tok // 64], tok % 64
            r = x[pg, sl, kv_head]
            if scale is not None:
                r = r * float(scale[pg, kv_head, sl])
            rows.append(r)
        return torch.stack(rows) if rows else torch.zeros((0, 128), dtype=torch.float64)

    return dec(case["k_cache"], case.get("k_scale")), dec(case["v_cache"], case.get("v_scale"))


def check_attn_vs_sdpa(case, tol=1e-12):
    """Oracle rows against torch's float64 scaled_dot_product_attention and logsumexp
    on the densely gathered K/V; query head qh reads KV head qh // G."""
    B, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    G = Hq // Hkv
    o, lse = oracle.attn_rows(case)
    if case.get("q_scale") is not None:
        q64 = (torch.from_numpy(case["q"]).view(torch.float8_e4m3fn).to(torch.float64)
               * torch.from_numpy(case["q_scale"]).to(torch.float64)[..., None])
    else:
        q64 = torch.from_numpy(case["q"].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    for b in range(B):
        if case["seq_lens"][b] <= 0:
            continue
        for kh in range(Hkv):
            K, V = dense_kv(case, b, kh)
            qg = q64[b, kh * G:(kh + 1) * G]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qg[None, :, None, :], K[None, None].expand(1, G, -1, -1),
                V[None, None].expand(1, G, -1, -1), scale=1 / math.sqrt(128))[0, :, 0]
            ref_lse = torch.logsumexp(qg @ K.T / math.sqrt(128), dim=-1)
            got = torch.from_numpy(o[b * Hq + kh * G:b * Hq + (kh + 1) * G])
            assert torch.allclose(got, ref, rtol=0, atol=tol), (b, kh, (got - ref).abs().max())
            gl = torch.from_numpy(lse[b * Hq + kh * G:b * Hq + (kh + 1) * G])
            assert torch.allclose(gl, ref_lse, rtol=0, atol=tol)


def check_attn_closed_forms():
    # L = 1: the output is v_0 and the LSE is the single scaled score.
    c = small_case([1], seed=3)
    o, lse = oracle.attn_rows(c)
    K, V = dense_kv(c, 0, 0)
    q = torch.from_numpy(c["q"].view(np.int16)).view(torch.bfloat16).to(torch.float64)[0]
    assert np.allclose(o, V[0].numpy()[None].repeat(8, 0), rtol=0, atol=0)
    assert np.allclose(lse, (q @ K[0]).numpy() / math.sqrt(128), rtol=0, atol=1e-13)
    # all-zero keys: uniform weights, O = mean(V), LSE = ln L
    c = small_case([150], seed=4)
    c["k_cache"][:] = 0
    o, lse = oracle.attn_rows(c)
    K, V = dense_kv(c, 0, 0)
    assert np.allclose(o, V.mean(0).numpy()[None].repeat(8, 0), rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(150), rtol=0, atol=1e-13)
    # identical keys: uniform weights again, LSE = s + ln L
    c = small_case([70], seed=5)
    pg = c["page_table"][0]
    for tok in range(70):
        c["k_cache"][pg[tok // 64], tok % 64, 0] = c["k_cache"][pg[0], 0, 0]
    o, lse = oracle.attn_rows(c)
    K, V = dense_kv(c, 0, 0)
    q = torch.from_numpy(c["q"].view(np.int16)).view(torch.bfloat16).to(torch.float64)[0]
    assert np.allclose(o, V.mean(0).numpy()[None].repeat(8, 0), rtol=0, atol=1e-12)
    assert np.allclose(lse, (q @ K[0]).numpy() / math.sqrt(128) + math.log(70), rtol=0, atol=1e-12)


def check_page_permutation_invariance():
    c = small_case([37, 300, 129], hkv=2, hq=16, seed=6, pool=30)
    o1, l1 = oracle.attn_rows(c)
    P = c["k_cache"].shape[0]
    perm = np.random.default_rng(1).permutation(P)
    inv = np.argsort(perm)
    c2 = dict(c)
    c2["k_cache"] = c["k_cache"][perm]
    c2["v_cache"] = c["v_cache"][perm]
    pt = c["page_table"].copy()
    pt[pt >= 0] = inv[pt[pt >= 0]]
    c2["page_table"] = pt
    o2, l2 = oracle.attn_rows(c2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def check_combine_equals_full(case, C, m, tol=1e-12):
    """Partials over the task map's ranges, merged, equal the unsplit softmax."""
    B, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    pb = oracle.plan(case["seq_lens"], Hkv, C, m)
    so, sl = oracle.attn_splits(pb, case)
    o, lse = oracle.combine(pb, so, sl, B, Hq, Hkv)
    fo, fl = oracle.attn_rows(case)
    fo = fo.reshape(B, Hq, 128)
    fl = fl.reshape(B, Hq)
    assert np.allclose(o, fo, rtol=0, atol=tol), np.abs(o - fo).max()
    fin = np.isfinite(fl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], fl[fin], rtol=0, atol=tol)
    return pb


def check_split_ranges(case, C, m):
    """Each partial equals plain attention over exactly its descriptor's tokens
    (a sub-sequence request built by slicing the page table)."""
    B, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    G = Hq // Hkv
    pb = oracle.plan(case["seq_lens"], Hkv, C, m)
    so, sl = oracle.attn_splits(pb, case)
    parsed = oracle.parse_plan(pb)
    for lst in parsed["lists"]:
        for (kh, b, c0, c1, s, _, _, _) in lst:
            L = int(case["seq_lens"][b])
            sub = dict(case)
            pt = np.full((1, c1 - c0), -1, dtype=np.int32)
            pt[0] = case["page_table"][b, c0:c1]
            sub["page_table"] = pt
            sub["seq_lens"] = np.array([min(64 * c1, L) - 64 * c0], dtype=np.int32)
            sub["q"] = case["q"][b:b + 1]
            rows = [(0, kh * G + j) for j in range(G)]
            o, lse = oracle.attn_rows(sub, rows)
            assert np.array_equal(o, so[s]) and np.array_equal(lse, sl[s])


def check_empty_request():
    c = small_case([0, 100], seed=7)
    o, lse = oracle.attn_rows(c)
    assert np.all(o[:8] == 0) and np.all(np.isneginf(lse[:8]))
    assert np.all(np.isfinite(lse[8:]))


# ------------------------------------------------------------------ several new tokens per request

def small_case_mt(lens, q_len, hkv=1, hq=8, dtype="bf16", seed=0, pool=None):
    w = wl.Workload("pin", len(lens), hq, hkv, dtype, seed, lens=list(lens), pool_pages=pool,
                    q_len=q_len)
    return wl.to_numpy_case(wl.make_case(w, device="cpu"))


def check_multitoken_vs_sdpa(case, tol=1e-12):
    """Rows of a q_len > 1 case against torch's float64 scaled_dot_product_attention
    with an explicit boolean mask: new token qi of request b may attend to key t
    iff t <= L_b - q_len + qi (the new tokens are the last q_len of the cache)."""
    B, Q, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    G = Hq // Hkv
    o, lse = oracle.attn_rows(case)
    o = o.reshape(B, Q, Hq, 128)
    lse = lse.reshape(B, Q, Hq)
    q64 = torch.from_numpy(case["q"].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    for b in range(B):
        L = int(case["seq_lens"][b])
        if L <= 0:
            assert np.all(o[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        allowed = torch.arange(L)[None, :] <= (L - Q + torch.arange(Q))[:, None]  # [Q, L]
        for kh in range(Hkv):
            K, V = dense_kv(case, b, kh)
            for qi in range(Q):
                qg = q64[b, qi, kh * G:(kh + 1) * G]
                got_o = o[b, qi, kh * G:(kh + 1) * G]
                got_l = lse[b, qi, kh * G:(kh + 1) * G]
                if not bool(allowed[qi].any()):
                    assert np.all(got_o == 0) and np.all(np.isneginf(got_l)), (b, qi)
                    continue
                mask = allowed[qi][None, None, None, :].expand(1, G, 1, L)
                ref = torch.nn.functional.scaled_dot_product_attention(
                    qg[None, :, None, :], K[None, None].expand(1, G, -1, -1),
                    V[None, None].expand(1, G, -1, -1), attn_mask=mask,
                    scale=1 / math.sqrt(128))[0, :, 0]
                sc = (qg @ K.T / math.sqrt(128)).masked_fill(~allowed[qi][None, :], float("-inf"))
                ref_lse = torch.logsumexp(sc, dim=-1)
                assert np.allclose(got_o, ref.numpy(), rtol=0, atol=tol), (b, qi, kh)
                assert np.allclose(got_l, ref_lse.numpy(), rtol=0, atol=tol), (b, qi, kh)


def check_multitoken_is_prefix_decode(case):
    """New token qi with q_len new tokens equals one-token decode of the same
    query over the first L - q_len + qi + 1 tokens (a shorter seq_lens)."""
    B, Q, Hq, _ = case["q"].shape
    o, lse = oracle.attn_rows(case)
    o = o.reshape(B, Q, Hq, 128)
    lse = lse.reshape(B, Q, Hq)
    for qi in range(Q):
        one = dict(case)
        one["q"] = np.ascontiguousarray(case["q"][:, qi])
        one["seq_lens"] = np.maximum(case["seq_lens"] - Q + qi + 1, 0).astype(np.int32)
        o1, l1 = oracle.attn_rows(one)
        assert np.array_equal(o1.reshape(B, Hq, 128), o[:, qi]), qi
        assert np.array_equal(l1.reshape(B, Hq), lse[:, qi]), qi


def check_multitoken_combine_equals_full(case, C, m, tol=1e-12):
    """Partials over a task map's ranges, merged per (request, new token, head),
    equal the unsplit causal softmax; tokens whose visible range ends before a
    descriptor's chunks contribute an empty partial there."""
    B, Q, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    pb = oracle.plan(case["seq_lens"], Hkv, C, m)
    so, sl = oracle.attn_splits(pb, case)
    assert so.shape[1:] == (Q, Hq // Hkv, 128)
    o, lse = oracle.combine(pb, so, sl, B, Hq, Hkv, q_len=Q)
    fo, fl = oracle.attn_rows(case)
    fo = fo.reshape(B, Q, Hq, 128)
    fl = fl.reshape(B, Q, Hq)
    assert np.allclose(o, fo, rtol=0, atol=tol), np.abs(o - fo).max()
    fin = np.isfinite(fl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], fl[fin], rtol=0, atol=tol)
    return pb, so, sl


def check_multitoken_split_ranges(case, C, m):
    """A partial of new token qi is plain attention over its descriptor's
    tokens clipped to qi's visible range (a sub-request cut from the page table)."""
    B, Q, Hq, _ = case["q"].shape
    Hkv = case["k_cache"].shape[2]
    G = Hq // Hkv
    pb = oracle.plan(case["seq_lens"], Hkv, C, m)
    so, sl = oracle.attn_splits(pb, case)
    for lst in oracle.parse_plan(pb)["lists"]:
        for (kh, b, c0, c1, s, _, _, _) in lst:
            L = int(case["seq_lens"][b])
            for qi in range(Q):
                vis = max(L - Q + qi + 1, 0)
                n = min(64 * c1, vis) - 64 * c0
                if n <= 0:
                    assert np.all(so[s, qi] == 0) and np.all(np.isneginf(sl[s, qi]))
                    continue
                sub = dict(case)
                sub["page_table"] = np.ascontiguousarray(case["page_table"][b:b + 1, c0:c1])
                sub["seq_lens"] = np.array([n], dtype=np.int32)
                sub["q"] = np.ascontiguousarray(case["q"][b:b + 1, qi])
                o, lse = oracle.attn_rows(sub, [(0, kh * G + j) for j in range(G)])
                assert np.array_equal(o, so[s, qi]) and np.array_equal(lse, sl[s, qi]), (s, qi)


def check_multitoken_short_requests():
    """L < q_len: the first q_len - L new tokens see nothing (O = 0, LSE = -inf);
    q_len = 1 reproduces the one-token layout."""
    c = small_case_mt([0, 2, 5, 70], 4, seed=21)
    o, lse = oracle.attn_rows(c)
    o = o.reshape(4, 4, 8, 128)
    lse = lse.reshape(4, 4, 8)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isneginf(lse[1, :2])) and np.all(np.isfinite(lse[1, 2:]))
    assert np.all(np.isfinite(lse[2:]))
    # L = 2, last new token: two keys; the first of the two new tokens sees only key 0
    K, V = dense_kv(c, 1, 0)
    assert np.allclose(o[1, 2], V[0].numpy()[None].repeat(8, 0), rtol=0, atol=0)
    one = small_case_mt([37, 300], 1, seed=22)
    assert one["q"].ndim == 3
