"""Seeded synthetic decode batches shaped like the pages' workloads.

This module only draws inputs: live KV lengths, page tables, and the BF16 /
FP8-e4m3 contents of Q and the paged K/V cache. It holds none of the attention
method's arithmetic and imports neither the CUDA library nor the oracle, so
both sides of a parity test can take their inputs from it.

Recipe (stated once here and in the design notes):
  * Lengths: fixed lists, or ``floor(exp(U[ln lo, ln hi]))`` clamped to
    [lo, hi] from ``numpy.random.default_rng(seed)``. With a total-token cap
    the lengths are scaled by cap / sum, floored and clamped to >= lo.
  * Page pool: a seeded permutation of ``pool_pages`` physical pages (the sum
    of the chunk counts when the workload names no pool). Request b takes the
    next n_b = ceil(L_b / 64) pages of the permutation. Table entries past n_b
    are -1 (never read by a correct kernel).
  * Q, K, V values: N(0, 1) drawn with ``torch.Generator(device)`` seeded from
    ``seed``, rounded to bfloat16. For an e4m3 cache each (token, KV head)
    128-vector x gets scale = amax|x| / 448 (1 when amax is 0) and codes
    e4m3(x / scale) by round-to-nearest-even; the scale is stored as float32 in
    [page][kv_head][slot] order.
  * An e4m3 Q (q_dtype "fp8") is quantised the same way per (request, query
    head), with its scale in a float32 [B, Hq] array.
  * Q/K/V of a large batch are drawn on the GPU; the oracle reads a host copy
    of the same bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
HEAD_DIM = 128
E4M3_MAX = 448.0
FOUR_M = 4 * 1024 * 1024


@dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    kv_dtype: str  # "bf16" or "fp8"
    seed: int
    lens: list | None = None          # fixed lengths
    loguniform: tuple | None = None   # (lo, hi)
    total_cap: int | None = None
    pool_pages: int | None = None
    num_ctas: int | None = None       # None: device default
    min_chunks: int = 2
    static_splits: int = 16
    q_dtype: str = "bf16"  # "bf16", or "fp8": e4m3 codes with one float32 scale per (request, head)
    q_len: int = 1         # new tokens per request (> 1: speculative verification rows)
    note: str = ""
    extra: dict = field(default_factory=dict)


# The five workloads the scope names (plus a batch of many short requests),
# and the six length mixes of the pages' decode-latency table (vLLM x HPC-Ops
# blog, Table 3), at the TP8-shard head shape (8 query heads, 1 KV head) and
# at the full Hy3 shape.
WORKLOADS = {
    "tiny": Workload("tiny", 4, 8, 1, "bf16", 0, lens=[37, 128, 300, 1000], pool_pages=64,
                     num_ctas=16, min_chunks=2,
                     note="batch 4, L={37,128,300,1000}, 8 Q / 1 KV head, 64-page pool, 16 CTAs, m=2"),
    "uniform": Workload("uniform", 16, 64, 8, "bf16", 1, lens=[4096] * 16, pool_pages=2048,
                        num_ctas=148,
                        note="batch 16 x 4096 tokens, 64 Q / 8 KV heads, 2048-page pool, 148 CTAs"),
    "mixed": Workload("mixed", 64, 64, 8, "bf16", 2, loguniform=(128, 65536),
                      note="batch 64, L log-uniform in [128, 65536], 64 Q / 8 KV heads, bf16"),
    "skew": Workload("skew", 32, 64, 8, "bf16", 3, lens=[131072] + [1024] * 31, static_splits=16,
                     note="batch 32: 1 x 131072 + 31 x 1024 tokens, 64 Q / 8 KV heads, bf16"),
    "fp8": Workload("fp8", 64, 64, 8, "fp8", 4, loguniform=(512, 262144), total_cap=FOUR_M,
                    note="batch 64, L log-uniform in [512, 262144] capped at 4M tokens, e4m3 KV"),
    "fp8q": Workload("fp8q", 64, 64, 8, "fp8", 4, loguniform=(512, 262144), total_cap=FOUR_M,
                     q_dtype="fp8",
                     note="the fp8 batch with e4m3 Q and a per-(request, head) Q scale"),
    # many short requests: every (KV head, request) pair is one two-chunk
    # descriptor, so per-descriptor costs (query staging, merge, partial
    # write) and the combine's per-pair work dominate instead of the KV stream
    "short": Workload("short", 1024, 64, 8, "bf16", 5, lens=[128] * 1024,
                      note="batch 1024 x 128 tokens, 64 Q / 8 KV heads, bf16 (8192 two-chunk descriptors)"),
}

TABLE3_MIXES = {
    "64x0.5K": [512] * 64,
    "64x4K": [4096] * 64,
    "32x0.125K+32x4K": [128] * 32 + [4096] * 32,
    "2x32K+30x4K": [32768] * 2 + [4096] * 30,
    "1x64K+15x4K": [65536] + [4096] * 15,
    "1x128K+31x4K": [131072] + [4096] * 31,
}


def table3_workload(mix: str, num_q_heads: int = 8, num_kv_heads: int = 1, seed: int = 10):
    lens = TABLE3_MIXES[mix]
    return Workload(f"t3:{mix}:{num_q_heads}/{num_kv_heads}", len(lens), num_q_heads, num_kv_heads,
                    "fp8", seed, lens=list(lens), note=f"decode-latency table mix {mix}, e4m3 KV")


def by_name(name: str) -> Workload:
    """A workload by name: one of WORKLOADS, or "t3:<mix>[:<Hq>/<Hkv>][:q8]" for a
    length mix of the decode-latency table (default 8 query / 1 KV head; ":q8"
    gives it an e4m3 query with per-head scales). A trailing ":qlen<N>" gives any
    of them N new tokens per request (causal verification rows)."""
    from dataclasses import replace
    if name in WORKLOADS:
        return WORKLOADS[name]
    if ":qlen" in name:
        base, n = name.rsplit(":qlen", 1)
        w = by_name(base)
        return replace(w, name=name, q_len=int(n), note=f"{w.note}; {int(n)} new tokens per request (causal)")
    parts = name.split(":")
    q8 = parts[-1] == "q8"
    if q8:
        parts = parts[:-1]
    if parts[0] == "t3" and len(parts) in (2, 3) and parts[1] in TABLE3_MIXES:
        hq, hkv = (8, 1) if len(parts) == 2 else (int(x) for x in parts[2].split("/"))
        w = table3_workload(parts[1], hq, hkv)
        if q8:
            w.q_dtype = "fp8"
            w.name += ":q8"
        return w
    raise KeyError(f"unknown workload {name!r}")


def draw_lengths(w: Workload) -> np.ndarray:
    if w.lens is not None:
        return np.asarray(w.lens, dtype=np.int64)
    lo, hi = w.loguniform
    rng = np.random.default_rng(w.seed)
    u = rng.uniform(math.log(lo), math.log(hi), size=w.batch)
    L = np.clip(np.floor(np.exp(u)), lo, hi).astype(np.int64)
    if w.total_cap is not None and L.sum() > w.total_cap:
        L = np.maximum(np.floor(L * (w.total_cap / L.sum())), lo).astype(np.int64)
    return L


def chunk_counts(lens) -> np.ndarray:
    lens = np.maximum(np.asarray(lens, dtype=np.int64), 0)
    return (lens + PAGE - 1) // PAGE


def draw_page_table(lens, pool_pages: int | None, seed: int, stride: int | None = None):
    """Seeded random page assignment. Returns (table int32 [B, stride], num_pages)."""
    n = chunk_counts(lens)
    need = int(n.sum())
    pool = max(need, 1) if pool_pages is None else int(pool_pages)
    if pool < need:
        raise ValueError(f"pool of {pool} pages is smaller than the {need} pages needed")
    rng = np.random.default_rng(seed + 7919)
    perm = rng.permutation(pool).astype(np.int32)
    stride = max(int(n.max()) if len(n) else 1, 1) if stride is None else stride
    table = np.full((len(n), stride), -1, dtype=np.int32)
    off = 0
    for b, nb in enumerate(n):
        table[b, :nb] = perm[off:off + nb]
        off += nb
    return table, pool


def _bf16_normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _fill_cache_bf16(num_pages, Hkv, gen, device, block_pages=2048):
    out = torch.empty((num_pages, PAGE, Hkv, HEAD_DIM), dtype=torch.bfloat16, device=device)
    for p0 in range(0, num_pages, block_pages):
        p1 = min(num_pages, p0 + block_pages)
        out[p0:p1] = _bf16_normal((p1 - p0, PAGE, Hkv, HEAD_DIM), gen, device)
    return out


def _fill_cache_e4m3(num_pages, Hkv, gen, device, block_pages=2048):
    codes = torch.empty((num_pages, PAGE, Hkv, HEAD_DIM), dtype=torch.float8_e4m3fn, device=device)
    scale = torch.empty((num_pages, Hkv, PAGE), dtype=torch.float32, device=device)
    for p0 in range(0, num_pages, block_pages):
        p1 = min(num_pages, p0 + block_pages)
        x = torch.randn((p1 - p0, PAGE, Hkv, HEAD_DIM), generator=gen, device=device,
                        dtype=torch.float32)
        amax = x.abs().amax(dim=-1, keepdim=True)
        s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        codes[p0:p1] = (x / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        scale[p0:p1] = s.squeeze(-1).permute(0, 2, 1)
    return codes, scale


def make_case(w: Workload, device="cpu", lens=None, pool_pages=None, stride=None) -> dict:
    """Draw one decode batch. Tensors live on ``device``.

    Returns a dict with q (bf16 [B,Hq,128], or float8_e4m3fn with q_scale float32
    [B,Hq] when the workload's q_dtype is "fp8"; [B,q_len,Hq,128] and
    [B,q_len,Hq] when the workload has q_len > 1), k_cache / v_cache (bf16 or
    float8_e4m3fn [pages,64,Hkv,128]), k_scale / v_scale (float32
    [pages,Hkv,64] or None), page_table (int32 [B,stride]), seq_lens (int32 [B]),
    num_pages, and the workload.
    """
    L = draw_lengths(w) if lens is None else np.asarray(lens, dtype=np.int64)
    table, num_pages = draw_page_table(L, w.pool_pages if pool_pages is None else pool_pages,
                                       w.seed, stride)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed) * 1000003 + 17)
    q_scale = None
    qshape = (len(L), w.num_q_heads, HEAD_DIM) if w.q_len == 1 else (len(L), w.q_len, w.num_q_heads, HEAD_DIM)
    if w.q_dtype == "fp8":
        x = torch.randn(qshape, generator=gen, device=device, dtype=torch.float32)
        amax = x.abs().amax(dim=-1, keepdim=True)
        s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        q = (x / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        q_scale = s.squeeze(-1).contiguous()
    else:
        q = _bf16_normal(qshape, gen, device)
    if w.kv_dtype == "fp8":
        k, ks = _fill_cache_e4m3(num_pages, w.num_kv_heads, gen, device)
        v, vs = _fill_cache_e4m3(num_pages, w.num_kv_heads, gen, device)
    else:
        k = _fill_cache_bf16(num_pages, w.num_kv_heads, gen, device)
        v = _fill_cache_bf16(num_pages, w.num_kv_heads, gen, device)
        ks = vs = None
    return dict(workload=w, q=q, q_scale=q_scale, k_cache=k, v_cache=v, k_scale=ks, v_scale=vs,
                page_table=torch.from_numpy(table).to(device),
                seq_lens=torch.from_numpy(L.astype(np.int32)).to(device),
                num_pages=num_pages)


def to_numpy_case(case: dict, requests=None) -> dict:
    """Host copy of a case as the oracle's numpy arrays (bf16 / e4m3 as raw bits).

    With ``requests`` given, only those requests' pages are copied: the copy
    holds a compact pool and a re-numbered page table for exactly those
    requests (rows keep their original order inside the subset).
    """
    q = case["q"]
    pt = case["page_table"].cpu().numpy()
    sl = case["seq_lens"].cpu().numpy()
    k, v, ks, vs = case["k_cache"], case["v_cache"], case["k_scale"], case["v_scale"]
    if requests is not None:
        req = np.asarray(requests, dtype=np.int64)
        n = chunk_counts(sl[req])
        pages = np.concatenate([pt[b, :nb] for b, nb in zip(req, n)]) if len(req) else np.zeros(0, np.int64)
        pages = pages.astype(np.int64)
        idx = torch.from_numpy(pages).to(k.device)
        k, v = k.index_select(0, idx), v.index_select(0, idx)
        if ks is not None:
            ks, vs = ks.index_select(0, idx), vs.index_select(0, idx)
        new_pt = np.full((len(req), max(int(n.max()) if len(n) else 1, 1)), -1, dtype=np.int32)
        off = 0
        for i, nb in enumerate(n):
            new_pt[i, :nb] = np.arange(off, off + nb, dtype=np.int32)
            off += nb
        pt, sl = new_pt, sl[req]
        q = q.index_select(0, torch.from_numpy(req).to(q.device))
        if case.get("q_scale") is not None:
            qs_sel = case["q_scale"].index_select(0, torch.from_numpy(req).to(q.device))

    def bits(t):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        if t.dtype == torch.float8_e4m3fn:
            return t.view(torch.uint8).numpy()
        return t.numpy()

    out = dict(q=bits(q), k_cache=bits(k), v_cache=bits(v), page_table=np.ascontiguousarray(pt),
               seq_lens=np.ascontiguousarray(sl.astype(np.int32)))
    if case.get("q_scale") is not None:
        qs = qs_sel if requests is not None else case["q_scale"]
        out["q_scale"] = qs.detach().cpu().numpy()
    if ks is not None:
        out["k_scale"] = ks.detach().cpu().numpy()
        out["v_scale"] = vs.detach().cpu().numpy()
    return out


def kv_bytes(lens, num_kv_heads: int, kv_dtype: str) -> int:
    """Bytes of live K and V (plus FP8 scales) for the given lengths."""
    tok = int(np.maximum(np.asarray(lens, dtype=np.int64), 0).sum())
    per = 2 * HEAD_DIM * (1 if kv_dtype == "fp8" else 2) + (8 if kv_dtype == "fp8" else 0)
    return tok * num_kv_heads * per


# ---------------------------------------------------------------- prologue inputs

def rope_table(max_pos: int, base: float = 10000.0) -> np.ndarray:
    """Rotary table float32 [max_pos, 128]: cos(p * base^(-2i/128)) for i < 64,
    then the matching sines (the model's precomputed rotary cache)."""
    i = np.arange(HEAD_DIM // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / HEAD_DIM)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def make_prologue_case(positions, num_q_heads, num_kv_heads, seed, device="cpu", max_pos=None,
                       slots=None, eps=1e-6):
    """Inputs of the fused prologue for tokens at the given positions: the QKV
    projection output (bf16 [T, Hq + 2*Hkv, 128], N(0,1)), per-dim RMSNorm
    weights (float32, 1 + 0.1 N(0,1)), the rotary table and the KV slots
    (int32 page*64 + offset, or -1 to skip)."""
    positions = np.asarray(positions, dtype=np.int32)
    T = len(positions)
    max_pos = int(positions.max()) + 1 if max_pos is None and T else (max_pos or 1)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 7919 + 3)
    H3 = num_q_heads + 2 * num_kv_heads
    qkv = torch.randn((T, H3, HEAD_DIM), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    rng = np.random.default_rng(seed + 11)
    qw = (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32)
    kw = (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32)
    if slots is None:
        slots = np.arange(T, dtype=np.int32)
    return dict(qkv=qkv, positions=torch.from_numpy(positions).to(device),
                cos_sin=torch.from_numpy(rope_table(max_pos)).to(device),
                q_weight=torch.from_numpy(qw).to(device), k_weight=torch.from_numpy(kw).to(device),
                slots=torch.from_numpy(np.asarray(slots, dtype=np.int32)).to(device), eps=eps,
                num_q_heads=num_q_heads, num_kv_heads=num_kv_heads)


def decode_slots(case: dict) -> np.ndarray:
    """Slot of each request's newest token (position L_b - 1) in a decode case."""
    pt = case["page_table"].cpu().numpy()
    L = case["seq_lens"].cpu().numpy().astype(np.int64)
    out = np.full(len(L), -1, dtype=np.int32)
    for b, n in enumerate(L):
        if n > 0:
            p = n - 1
            out[b] = pt[b, p // PAGE] * PAGE + p % PAGE
    return out
