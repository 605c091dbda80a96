"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/hpc_decode.h declares, and rejects bad arguments on the host
before any CUDA work (fake, never-dereferenced pointers)."""
import ctypes
import os
import re

import pytest

import oracle
from load_balanced_paged_02_gb300 import _build
from load_balanced_paged_02_gb300 import binding as hb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hpc_decode.h")
FAKE = ctypes.c_void_p(0x10000)      # 256-byte aligned, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x10004)  # not 16-byte aligned


@pytest.fixture(scope="module")
def L():
    _build.build()
    return hb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(hpc_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("hpc_decode_plan", "hpc_decode_plan_static", "hpc_decode_attn",
                     "hpc_decode_combine", "hpc_decode_step_host", "hpc_decode_read_error"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} not exported"
    assert set(declared_functions()) == set(hb.SIGNATURES), "binding and header disagree"


def test_plan_bytes_match_layout(L):
    for B, H, C in [(1, 1, 1), (4, 1, 16), (64, 8, 152), (16384, 1, 5000), (7, 3, 999)]:
        assert L.hpc_decode_plan_bytes(B, H, C) == 4 * oracle.layout(B, H, C)["total"]
        assert L.hpc_decode_split_capacity(B, H, C) == H * B + C - 1
    assert L.hpc_decode_plan_bytes(0, 1, 1) == 0
    assert L.hpc_decode_plan_bytes(16385, 1, 1) == 0
    assert L.hpc_decode_plan_bytes(1, 257, 1) == 0
    assert L.hpc_decode_plan_bytes(1, 1, 0) == 0


def test_auto_engine_choice(L):
    """Warp-level kernels for one and two new tokens, tcgen05 from three, for
    both cache dtypes; bad arguments give 0."""
    for kvd in (hb.KV_BF16, hb.KV_FP8_E4M3):
        assert [L.hpc_decode_attn_multi_auto_engine(kvd, q) for q in range(1, 9)] == \
            [hb.ENGINE_MMA_SYNC] * 2 + [hb.ENGINE_TCGEN05] * 6
        assert L.hpc_decode_attn_multi_auto_engine(kvd, 0) == 0
        assert L.hpc_decode_attn_multi_auto_engine(kvd, 9) == 0
    assert L.hpc_decode_attn_multi_auto_engine(7, 3) == 0


def test_status_strings(L):
    for code in range(6):
        assert L.hpc_status_string(code)
    assert L.hpc_status_string(99) == b"unknown status"


def _attn(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, dt=0, pages=16, pt=FAKE, stride=4, sl=FAKE,
             B=2, Hq=8, Hkv=1, D=128, P=64, plan=None, so=FAKE, slse=FAKE)
    a.update(kw)
    return L.hpc_decode_attn(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["dt"], a["pages"], a["pt"],
                             a["stride"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"], a["plan"],
                             a["so"], a["slse"], None)


def test_attn_rejects_unsupported_shapes(L):
    assert _attn(L, D=64) == 2
    assert _attn(L, P=16) == 2
    assert _attn(L, Hq=16, Hkv=1) == 2
    assert _attn(L, dt=7) == 2


def test_attn_rejects_bad_arguments(L):
    plan = hb.PlanStruct(FAKE.value, 1 << 20, 2, 1, 4, 2, 0, 10)
    assert _attn(L, q=None, plan=ctypes.byref(plan)) == 1
    assert _attn(L, q=FAKE_ODD, plan=ctypes.byref(plan)) == 1
    assert _attn(L, dt=1, plan=ctypes.byref(plan)) == 1          # e4m3 without scales
    assert _attn(L, plan=None) == 1
    wrong = hb.PlanStruct(FAKE.value, 1 << 20, 3, 1, 4, 2, 0, 10)  # batch mismatch
    assert _attn(L, plan=ctypes.byref(wrong)) == 1
    small = hb.PlanStruct(FAKE.value, 8, 2, 1, 4, 2, 0, 10)        # buffer too small
    assert _attn(L, plan=ctypes.byref(small)) == 1
    assert _attn(L, pages=0, plan=ctypes.byref(plan)) == 1


def test_attn_q8_rejects_bad_arguments(L):
    plan = hb.PlanStruct(FAKE.value, 1 << 20, 2, 1, 4, 2, 0, 10)
    args = dict(q8=FAKE, qs=FAKE, k=FAKE, v=FAKE, ks=FAKE, vs=FAKE, pages=16, pt=FAKE, stride=4, sl=FAKE,
                B=2, Hq=8, Hkv=1, D=128, P=64, plan=ctypes.byref(plan), so=FAKE, slse=FAKE)

    def call(**kw):
        a = dict(args, **kw)
        return L.hpc_decode_attn_q8(a["q8"], a["qs"], a["k"], a["v"], a["ks"], a["vs"], a["pages"], a["pt"],
                                    a["stride"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"],
                                    a["plan"], a["so"], a["slse"], None)
    assert call(qs=None) == 1
    assert call(qs=FAKE_ODD) == 1
    assert call(ks=None) == 1
    assert call(D=64) == 2


def test_attn_ex_rejects_bad_arguments(L):
    """hpc_decode_attn_ex: unknown flag bits, q_len, engine and query-scale
    combinations are refused on the host."""
    plan = hb.PlanStruct(FAKE.value, 1 << 20, 2, 1, 4, 2, 0, 10)
    args = dict(q=FAKE, qs=None, ql=1, k=FAKE, v=FAKE, ks=None, vs=None, dt=0, pages=16, pt=FAKE, stride=4,
                sl=FAKE, B=2, Hq=8, Hkv=1, D=128, P=64, plan=ctypes.byref(plan), so=FAKE, slse=FAKE, eng=0,
                flags=hb.ATTN_EARLY_KV)

    def call(**kw):
        a = dict(args, **kw)
        return L.hpc_decode_attn_ex(a["q"], a["qs"], a["ql"], a["k"], a["v"], a["ks"], a["vs"], a["dt"],
                                    a["pages"], a["pt"], a["stride"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["D"],
                                    a["P"], a["plan"], a["so"], a["slse"], a["eng"], a["flags"], None)
    assert call(flags=4) == 1
    assert call(flags=-1) == 1
    # the failure-path test flag: one new token on the warp-level kernel only
    assert call(flags=hb.ATTN_TEST_WAIT_EXPIRY, ql=2) == 2
    assert call(flags=hb.ATTN_TEST_WAIT_EXPIRY, ql=3) == 2
    assert call(flags=hb.ATTN_TEST_WAIT_EXPIRY, eng=hb.ENGINE_TCGEN05) == 2
    assert call(ql=0) == 1
    assert call(ql=9) == 1
    assert call(eng=3) == 1
    assert call(qs=FAKE) == 2                            # a query scale with a bf16 cache
    assert call(qs=FAKE, dt=1, ks=FAKE, vs=FAKE, ql=2) == 1  # e4m3 query is one token per request
    assert call(q=None) == 1
    assert call(D=64) == 2


def test_step_graph_rejects_bad_arguments(L):
    """hpc_decode_step_graph_*: argument checks before any CUDA call."""
    handle = ctypes.c_void_p(1234)
    args = [FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, None, 0, 16, 2, 8, 1, 128, 64, 4, 2, FAKE, 1 << 30, FAKE, None]

    def create(*over, graph=ctypes.byref(handle)):
        a = list(args)
        for i, v in over:
            a[i] = v
        return L.hpc_decode_step_graph_create(*a, graph)
    assert create(graph=None) == 1
    assert create((0, None)) == 1 and handle.value is None           # no h_q; *graph cleared
    assert create((13, 64)) == 2                                       # head_dim
    assert create((8, 7)) == 2                                         # kv dtype
    assert create((17, FAKE_ODD)) == 1                                 # workspace alignment
    assert create((18, 16)) == 3                                       # workspace too small
    assert L.hpc_decode_step_graph_launch(None, None) == 1
    assert L.hpc_decode_step_graph_destroy(None) == 0


def test_plan_rejects_bad_arguments(L):
    p = hb.PlanStruct(FAKE.value, 1 << 20, 0, 0, 0, 0, 0, 0)
    assert L.hpc_decode_plan(None, 4, 1, 16, 2, ctypes.byref(p), None) == 1
    assert L.hpc_decode_plan(FAKE, 0, 1, 16, 2, ctypes.byref(p), None) == 1
    assert L.hpc_decode_plan(FAKE, 4, 1, 16, -1, ctypes.byref(p), None) == 1
    assert L.hpc_decode_plan(FAKE, 4, 1, 0, 2, ctypes.byref(p), None) == 1
    small = hb.PlanStruct(FAKE.value, 64, 0, 0, 0, 0, 0, 0)
    assert L.hpc_decode_plan(FAKE, 4, 1, 16, 2, ctypes.byref(small), None) == 3
    odd = hb.PlanStruct(FAKE_ODD.value, 1 << 20, 0, 0, 0, 0, 0, 0)
    assert L.hpc_decode_plan(FAKE, 4, 1, 16, 2, ctypes.byref(odd), None) == 1
    assert L.hpc_decode_plan_static(FAKE, 4, 1, 0, ctypes.byref(p), None) == 1
    assert L.hpc_decode_plan_static(FAKE, 4, 1, 16, ctypes.byref(small), None) == 3


def test_combine_and_step_reject_bad_arguments(L):
    plan = hb.PlanStruct(FAKE.value, 1 << 20, 2, 1, 4, 2, 0, 10)
    assert L.hpc_decode_combine(ctypes.byref(plan), FAKE, FAKE, FAKE, None, 2, 8, 1, 64, None) == 2
    assert L.hpc_decode_combine(ctypes.byref(plan), None, FAKE, FAKE, None, 2, 8, 1, 128, None) == 1
    assert L.hpc_decode_combine(None, FAKE, FAKE, FAKE, None, 2, 8, 1, 128, None) == 1
    ws = L.hpc_decode_step_workspace_bytes(2, 8, 1, 4, 4)
    assert ws > 0 and ws % 256 == 0
    args = [FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, None, 0, 16, 2, 8, 1, 128, 64, 4, 2, FAKE]
    assert L.hpc_decode_step_host(*args, ws - 1, FAKE, None, None) == 3
    assert L.hpc_decode_step_host(*args[:-1], FAKE_ODD, ws, FAKE, None, None) == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(hb, "_LIB", None)
    monkeypatch.setattr(hb._build, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(hb.HpcError):
        hb.lib()


def test_rope_norm_rejects_bad_arguments(L):
    """Every call here is refused on the host (or has no tokens), so nothing
    is launched with the fake pointers."""
    def call(**kw):
        a = dict(qkv=FAKE, positions=FAKE, cos_sin=FAKE, max_pos=4096, q_weight=FAKE, k_weight=FAKE, eps=1e-6,
                 slots=FAKE, num_tokens=4, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                 q_out=FAKE, q_scale=None, k_cache=FAKE, v_cache=FAKE, k_scale=None, v_scale=None,
                 kv_dtype=hb.KV_BF16, num_pages=16, err=None)
        a.update(kw)
        return L.hpc_rope_norm(a["qkv"], a["positions"], a["cos_sin"], a["max_pos"], a["q_weight"],
                               a["k_weight"], a["eps"], a["slots"], a["num_tokens"], a["num_q_heads"],
                               a["num_kv_heads"], a["head_dim"], a["page_size"], a["q_out"], a["q_scale"],
                               a["k_cache"], a["v_cache"], a["k_scale"], a["v_scale"], a["kv_dtype"],
                               a["num_pages"], a["err"], None)
    assert call(head_dim=64) == 2
    assert call(page_size=32) == 2
    assert call(kv_dtype=7) == 2
    for bad in (dict(num_tokens=-1), dict(num_q_heads=0), dict(num_kv_heads=0), dict(num_kv_heads=257),
                dict(max_pos=0), dict(num_pages=0), dict(eps=float("nan")), dict(eps=-1.0), dict(qkv=None),
                dict(positions=None), dict(slots=None), dict(k_cache=None), dict(qkv=FAKE_ODD),
                dict(q_out=FAKE_ODD), dict(kv_dtype=hb.KV_FP8_E4M3), dict(kv_dtype=hb.KV_FP8_E4M3, k_scale=FAKE)):
        assert call(**bad) == 1, bad
    # no tokens: valid and nothing to do
    assert call(num_tokens=0) == 0
    assert call(num_tokens=0, kv_dtype=hb.KV_FP8_E4M3, k_scale=FAKE, v_scale=FAKE) == 0


def test_noalloc_refuses_before_any_work(L):
    """hpc_decode_noalloc runs every check of plan, attention and combine
    before its first launch (fake pointers: nothing may be enqueued)."""
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ks=None, vs=None, dt=0, pages=1000, pt=FAKE, stride=8, sl=FAKE, B=24,
                 Hq=64, Hkv=8, D=128, P=64, C=152, m=2, out=FAKE, lse=None)
        a.update(kw)
        return L.hpc_decode_noalloc(a["q"], a["k"], a["v"], a["ks"], a["vs"], a["dt"], a["pages"], a["pt"],
                                    a["stride"], a["sl"], a["B"], a["Hq"], a["Hkv"], a["D"], a["P"], a["C"],
                                    a["m"], a["out"], a["lse"], None)
    assert call(B=4096) == 3                      # beyond the fixed array
    assert call(D=64) == 2
    assert call(P=32) == 2
    assert call(Hq=32) == 2
    assert call(dt=7) == 2
    for bad in (dict(q=None), dict(sl=None), dict(pt=None), dict(out=None), dict(q=FAKE_ODD),
                dict(out=ctypes.c_void_p(0x10002)), dict(m=-1), dict(pages=0), dict(stride=0),
                dict(dt=1), dict(dt=1, ks=FAKE), dict(B=0), dict(C=0)):
        assert call(**bad) == 1, bad


def test_suggest_num_ctas_refuses_bad_arguments(L):
    """Host-side checks of hpc_decode_suggest_num_ctas (0 for bad arguments)."""
    import numpy as np
    sl = np.full(8, 100, dtype=np.int32)
    p = ctypes.c_void_p(sl.ctypes.data)
    assert L.hpc_decode_suggest_num_ctas(None, 8, 8, 2, 0, 1) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 0, 8, 2, 0, 1) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 8, 0, 2, 0, 1) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 8, 8, -1, 0, 1) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 8, 8, 2, 7, 1) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 8, 8, 2, 0, 0) == 0
    assert L.hpc_decode_suggest_num_ctas(p, 8, 8, 2, 0, 9) == 0
