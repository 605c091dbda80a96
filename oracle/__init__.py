"""Float64 CPU oracle for load-balanced paged GQA decode attention.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library (``load_balanced_paged_02_gb300``) and never imports it.

The arithmetic lives in ``hpc_oracle.c`` (plain C, float64, optional OpenMP
over independent rows). This module only compiles it with gcc, loads it with
ctypes and marshals numpy arrays. ``parse_plan`` reads the task-map byte layout
that ``hpc_oracle.c`` defines, so that tests can check invariants of a map.

Sources: the HPC-Ops/SGLang blog, section "Scheduling around live KV work",
and the vLLM x HPC-Ops blog, sub-section "解决方案：按步负载均衡的 decode 调度器"
(assign -> compute -> combine).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hpc_oracle.c")
LIB = os.path.join(HERE, "libhpc_oracle.so")

CHUNK_TOKENS = 64
HEAD_DIM = 128
HDR_INTS = 16
TASK_INTS = 8
HDR_FIELDS = (
    "total_chunks", "bucket", "used_ctas", "total_splits", "num_ctas", "batch",
    "num_kv_heads", "min_chunks", "max_tasks", "mode", "chunks_per_head",
    "chunk_tokens", "error",
)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile hpc_oracle.c into libhpc_oracle.so with gcc (OpenMP if available)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        _lib = load_library(LIB)
        return _lib


def load_library(path: str):
    """Load and type a compiled oracle library (the default one, or a test copy)."""
    L = ctypes.CDLL(path)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    ci = ctypes.c_int
    L.oracle_plan_ints.argtypes = [ci, ci, ci]
    L.oracle_plan_ints.restype = ctypes.c_longlong
    L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_to_f64.restype = ctypes.c_double
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f64.restype = ctypes.c_double
    L.oracle_num_threads.restype = ci
    L.oracle_set_num_threads.argtypes = [ci]
    L.oracle_plan.argtypes = [i32p, ci, ci, ci, ci, i32p, ctypes.c_longlong]
    L.oracle_plan_static.argtypes = [i32p, ci, ci, ci, i32p, ctypes.c_longlong]
    kv = [vp, vp, vp, vp, vp, vp, ci, ci, i32p, ci, i32p, ci, ci, ci, ci]
    L.oracle_attn_rows.argtypes = kv + [ci, i32p, f64p, f64p]
    L.oracle_attn_splits.argtypes = [i32p] + kv + [f64p, f64p]
    L.oracle_combine.argtypes = [i32p, f64p, f64p, ci, ci, ci, ci, f64p, f64p]
    L.oracle_rope_norm.argtypes = [ctypes.POINTER(ctypes.c_uint16), i32p, ctypes.POINTER(ctypes.c_float), ci,
                                   ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                                   ctypes.c_double, ci, ci, ci, f64p, f64p, f64p]
    for f in ("oracle_plan", "oracle_plan_static", "oracle_attn_rows", "oracle_attn_splits",
              "oracle_combine", "oracle_rope_norm"):
        getattr(L, f).restype = ci
    return L


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _vp(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(int(code) & 0xFF)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits) & 0xFFFF)


def plan_ints(batch: int, num_kv_heads: int, num_ctas: int) -> int:
    return int(_load().oracle_plan_ints(batch, num_kv_heads, num_ctas))


def plan(seq_lens, num_kv_heads: int, num_ctas: int, min_chunks: int) -> np.ndarray:
    """Load-balanced task map (int32 array in the canonical layout)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.shape[0]
    out = np.empty(plan_ints(B, num_kv_heads, num_ctas), dtype=np.int32)
    rc = _load().oracle_plan(_p(sl, ctypes.c_int32), B, num_kv_heads, num_ctas, min_chunks,
                             _p(out, ctypes.c_int32), out.size)
    if rc:
        raise ValueError(f"oracle_plan failed ({rc})")
    return out


def plan_static(seq_lens, num_kv_heads: int, num_splits: int) -> np.ndarray:
    """Static split-KV task map with a fixed split count per (kv head, request)."""
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.shape[0]
    out = np.empty(plan_ints(B, num_kv_heads, num_kv_heads * B * num_splits), dtype=np.int32)
    rc = _load().oracle_plan_static(_p(sl, ctypes.c_int32), B, num_kv_heads, num_splits,
                                    _p(out, ctypes.c_int32), out.size)
    if rc:
        raise ValueError(f"oracle_plan_static failed ({rc})")
    return out


def layout(batch: int, num_kv_heads: int, num_ctas: int) -> dict:
    """Offsets (in int32 units) of the sections of the task-map layout."""
    max_tasks = num_kv_heads * batch + 2 * num_ctas
    tasks = (HDR_INTS + num_ctas + 1 + 7) // 8 * 8
    nsplit = tasks + max_tasks * TASK_INTS
    split0 = nsplit + num_kv_heads * batch
    return dict(cta_off=HDR_INTS, tasks=tasks, nsplit=nsplit, split0=split0,
                total=split0 + num_kv_heads * batch, max_tasks=max_tasks)


def parse_plan(buf) -> dict:
    """Split a task-map buffer into its header, per-CTA descriptor lists and pair tables."""
    buf = np.asarray(buf, dtype=np.int32)
    hdr = {k: int(buf[i]) for i, k in enumerate(HDR_FIELDS)}
    B, Hkv, C = hdr["batch"], hdr["num_kv_heads"], hdr["num_ctas"]
    lay = layout(B, Hkv, C)
    cta_off = buf[lay["cta_off"]:lay["cta_off"] + C + 1].copy()
    tasks = buf[lay["tasks"]:lay["nsplit"]].reshape(lay["max_tasks"], TASK_INTS)
    lists = []
    for j in range(C):
        lst, k = [], int(cta_off[j])
        while tasks[k, 0] >= 0:
            lst.append(tuple(int(x) for x in tasks[k]))
            k += 1
        lists.append(lst)
    return dict(header=hdr, cta_off=cta_off, tasks=tasks.copy(), lists=lists,
                pair_nsplit=buf[lay["nsplit"]:lay["split0"]].copy(),
                pair_split0=buf[lay["split0"]:lay["total"]].copy(), layout=lay)


def _kv_args(case):
    fp8 = case["k_cache"].dtype == np.uint8
    kc = np.ascontiguousarray(case["k_cache"])
    vc = np.ascontiguousarray(case["v_cache"])
    ks = vs = None
    if fp8:
        ks = np.ascontiguousarray(case["k_scale"], dtype=np.float32)
        vs = np.ascontiguousarray(case["v_scale"], dtype=np.float32)
    qs = None
    if case.get("q_scale") is not None:
        q = np.ascontiguousarray(case["q"], dtype=np.uint8)
        qs = np.ascontiguousarray(case["q_scale"], dtype=np.float32)
    else:
        q = np.ascontiguousarray(case["q"], dtype=np.uint16)
    pt = np.ascontiguousarray(case["page_table"], dtype=np.int32)
    sl = np.ascontiguousarray(case["seq_lens"], dtype=np.int32)
    # q is [B, Hq, 128] (one new token per request) or [B, q_len, Hq, 128]
    B, Hq = q.shape[0], q.shape[-2]
    q_len = q.shape[1] if q.ndim == 4 else 1
    Hkv = kc.shape[2]
    keep = (q, qs, kc, vc, ks, vs, pt, sl)
    args = [_vp(q), _vp(qs), _vp(kc), _vp(vc), _vp(ks), _vp(vs), int(fp8), int(kc.shape[0]),
            _p(pt, ctypes.c_int32), int(pt.shape[1]), _p(sl, ctypes.c_int32), B, Hq, Hkv, q_len]
    return args, keep, B, Hq, Hkv, q_len


def attn_rows(case: dict, rows=None):
    """Full-sequence attention (float64) for the given (b, r) rows, or all rows.

    ``case`` holds numpy arrays: q (uint16 bf16 bits [B,Hq,128], or uint8 e4m3
    codes with q_scale float32 [B,Hq]; with several new tokens per request
    [B,q_len,Hq,128] and [B,q_len,Hq]), k_cache and
    v_cache (uint16 bf16 bits or uint8 e4m3 codes, [pages,64,Hkv,128]),
    k_scale/v_scale (float32 [pages,Hkv,64], e4m3 only), page_table
    (int32 [B, stride]) and seq_lens (int32 [B], counting the new tokens).
    A row is (b, qi * Hq + qh); new token qi attends causally to tokens
    [0, L_b - q_len + qi]. Returns (o [n,128] float64, lse [n] float64), all
    rows in (b, qi, qh) order when ``rows`` is None.
    """
    args, keep, B, Hq, Hkv, q_len = _kv_args(case)
    if rows is None:
        n, rp = B * q_len * Hq, None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n, rp = r.shape[0], _p(r, ctypes.c_int32)
        keep = keep + (r,)
    o = np.zeros((n, HEAD_DIM), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _load().oracle_attn_rows(*args, n, rp, _p(o, ctypes.c_double), _p(lse, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle_attn_rows failed ({rc})")
    return o, lse


def attn_splits(plan_buf, case: dict):
    """Per-descriptor partial outputs and LSE of a task map (float64).

    Returns (split_o [total_splits, G, 128], split_lse [total_splits, G]); with
    a 4-D q, (split_o [total_splits, q_len, G, 128], split_lse [total_splits, q_len, G]).
    """
    pb = np.ascontiguousarray(plan_buf, dtype=np.int32)
    args, keep, B, Hq, Hkv, q_len = _kv_args(case)
    G = Hq // Hkv
    S = max(int(pb[3]), 1)
    so = np.zeros((S, q_len, G, HEAD_DIM), dtype=np.float64)
    sl = np.zeros((S, q_len, G), dtype=np.float64)
    rc = _load().oracle_attn_splits(_p(pb, ctypes.c_int32), *args, _p(so, ctypes.c_double),
                                    _p(sl, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle_attn_splits failed ({rc})")
    if np.asarray(case["q"]).ndim == 3:
        so, sl = so[:, 0], sl[:, 0]
    return so[: int(pb[3])], sl[: int(pb[3])]


def combine(plan_buf, split_o, split_lse, batch: int, num_q_heads: int, num_kv_heads: int,
            q_len: int | None = None):
    """Merge partials into [B, Hq, 128] outputs and [B, Hq] LSE (float64);
    with ``q_len`` given, into [B, q_len, Hq, 128] and [B, q_len, Hq]."""
    pb = np.ascontiguousarray(plan_buf, dtype=np.int32)
    G = num_q_heads // num_kv_heads
    n = 1 if q_len is None else int(q_len)
    so = np.ascontiguousarray(split_o, dtype=np.float64).reshape(-1, n, G, HEAD_DIM)
    sl = np.ascontiguousarray(split_lse, dtype=np.float64).reshape(-1, n, G)
    if so.shape[0] == 0:
        so = np.zeros((1, n, G, HEAD_DIM))
        sl = np.zeros((1, n, G))
    o = np.zeros((batch, n, num_q_heads, HEAD_DIM), dtype=np.float64)
    lse = np.zeros((batch, n, num_q_heads), dtype=np.float64)
    rc = _load().oracle_combine(_p(pb, ctypes.c_int32), _p(so, ctypes.c_double),
                                _p(sl, ctypes.c_double), batch, num_q_heads, num_kv_heads, n,
                                _p(o, ctypes.c_double), _p(lse, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle_combine failed ({rc})")
    if q_len is None:
        return o[:, 0], lse[:, 0]
    return o, lse


def rope_norm(qkv_bits, positions, cos_sin, q_weight, k_weight, eps, num_q_heads, num_kv_heads):
    """Fused prologue in float64: RMS QK-norm then rotary embedding on Q and K,
    V passed through. qkv_bits: uint16 bf16 bits [T, Hq + 2*Hkv, 128].
    Returns (q [T,Hq,128], k [T,Hkv,128], v [T,Hkv,128]) float64, before rounding."""
    x = np.ascontiguousarray(qkv_bits, dtype=np.uint16)
    T = x.shape[0]
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    qw = np.ascontiguousarray(q_weight, dtype=np.float32)
    kw = np.ascontiguousarray(k_weight, dtype=np.float32)
    q = np.zeros((T, num_q_heads, HEAD_DIM))
    k = np.zeros((T, num_kv_heads, HEAD_DIM))
    v = np.zeros((T, num_kv_heads, HEAD_DIM))
    rc = _load().oracle_rope_norm(_p(x, ctypes.c_uint16), _p(pos, ctypes.c_int32), _p(cs, ctypes.c_float),
                                  cs.shape[0], _p(qw, ctypes.c_float), _p(kw, ctypes.c_float), float(eps), T,
                                  num_q_heads, num_kv_heads, _p(q, ctypes.c_double), _p(k, ctypes.c_double),
                                  _p(v, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle_rope_norm failed ({rc})")
    return q, k, v
