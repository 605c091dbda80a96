"""Thin ctypes binding of libhpcdecode (include/hpc_decode.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of the library. Torch tensors supply device pointers and the current
CUDA stream; nothing here computes attention, and every call raises HpcError
when the library is missing or returns a non-OK status.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

KV_BF16 = 0
KV_FP8_E4M3 = 1
ENGINE_AUTO, ENGINE_MMA_SYNC, ENGINE_TCGEN05 = 0, 1, 2
ATTN_EARLY_KV = 1  # flags of hpc_decode_attn_ex
ATTN_TEST_WAIT_EXPIRY = 2
HEAD_DIM = 128
PAGE = 64
GROUP = 8

_STATUS = {0: "HPC_OK", 1: "HPC_ERR_INVALID_ARG", 2: "HPC_ERR_UNSUPPORTED",
           3: "HPC_ERR_WORKSPACE_TOO_SMALL", 4: "HPC_ERR_CUDA", 5: "HPC_ERR_DEVICE_CHECK"}

# Every function include/hpc_decode.h declares: name -> (restype, argtypes).
_i = ctypes.c_int
_sz = ctypes.c_size_t
_vp = ctypes.c_void_p


class HpcError(RuntimeError):
    def __init__(self, where, status=None, detail=""):
        self.status = status
        name = _STATUS.get(status, str(status)) if status is not None else ""
        super().__init__(f"{where}: {name} {detail}".strip())


class PlanStruct(ctypes.Structure):
    _fields_ = [("buf", _vp), ("bytes", _sz), ("batch", _i), ("num_kv_heads", _i),
                ("num_ctas", _i), ("min_chunks", _i), ("mode", _i), ("max_tasks", _i)]


_P = ctypes.POINTER(PlanStruct)
SIGNATURES = {
    "hpc_decode_plan_bytes": (_sz, [_i, _i, _i]),
    "hpc_decode_split_capacity": (_sz, [_i, _i, _i]),
    "hpc_decode_default_num_ctas": (_i, [_i]),
    "hpc_decode_suggest_num_ctas": (_i, [_vp, _i, _i, _i, _i, _i]),
    "hpc_decode_attn_multi_auto_engine": (_i, [_i, _i]),
    "hpc_decode_plan": (_i, [_vp, _i, _i, _i, _i, _P, _vp]),
    "hpc_decode_plan_static": (_i, [_vp, _i, _i, _i, _P, _vp]),
    "hpc_decode_attn": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i, _i, _i, _i, _P,
                             _vp, _vp, _vp]),
    "hpc_decode_attn_q8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _i, _i, _P,
                                _vp, _vp, _vp]),
    "hpc_decode_attn_multi": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                   _P, _vp, _vp, _vp]),
    "hpc_decode_attn_multi_engine": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i, _i, _i,
                                          _i, _P, _vp, _vp, _i, _vp]),
    "hpc_decode_attn_ex": (_i, [_vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                _P, _vp, _vp, _i, _i, _vp]),
    "hpc_decode_combine": (_i, [_P, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "hpc_decode_combine_multi": (_i, [_P, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "hpc_rope_norm": (_i, [_vp, _vp, _vp, _i, _vp, _vp, ctypes.c_float, _vp, _i, _i, _i, _i, _i, _vp, _vp,
                           _vp, _vp, _vp, _vp, _i, _i, _vp, _vp]),
    "hpc_decode_step_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "hpc_decode_step_host": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                  _i, _i, _vp, _sz, _vp, _vp, _vp]),
    "hpc_decode_step_graph_create": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                                          _i, _vp, _sz, _vp, _vp, ctypes.POINTER(_vp)]),
    "hpc_decode_step_graph_launch": (_i, [_vp, _vp]),
    "hpc_decode_step_graph_destroy": (_i, [_vp]),
    "hpc_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                _i, _vp, _vp, _vp]),
    "hpc_decode_read_error": (_i, [_P, ctypes.POINTER(_i)]),
    "hpc_status_string": (ctypes.c_char_p, [_i]),
}

_lock = threading.Lock()
_LIB = None


def build(force: bool = False) -> str:
    """Compile libhpcdecode.so for sm_103a in-tree (nvcc)."""
    return _build.build(force=force)


def lib():
    """The loaded library; raises HpcError if it has not been built."""
    global _LIB
    with _lock:
        if _LIB is None:
            if not os.path.exists(_build.LIB_PATH):
                raise HpcError("libhpcdecode.so", detail="is not built; call "
                               "load_balanced_paged_02_gb300.build() (needs nvcc)")
            L = ctypes.CDLL(_build.LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _LIB = L
        return _LIB


def _check(name, rc):
    if rc != 0:
        msg = lib().hpc_status_string(rc).decode()
        raise HpcError(name, rc, f"({msg})")


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda_i32(t, what):
    if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
        raise HpcError(what, detail="must be a contiguous int32 CUDA tensor")
    return t


def kv_dtype_of(cache: torch.Tensor) -> int:
    if cache.dtype == torch.bfloat16:
        return KV_BF16
    if cache.dtype in (torch.float8_e4m3fn, torch.uint8):
        return KV_FP8_E4M3
    raise HpcError("k_cache", detail=f"unsupported dtype {cache.dtype}")


def sm_count(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def auto_engine(kv_dtype: int, q_len: int) -> int:
    """ENGINE_MMA_SYNC or ENGINE_TCGEN05: the kernel ENGINE_AUTO runs."""
    e = lib().hpc_decode_attn_multi_auto_engine(kv_dtype, q_len)
    if e == 0:
        raise HpcError("hpc_decode_attn_multi_auto_engine", detail=f"kv_dtype {kv_dtype}, q_len {q_len}")
    return e


def default_num_ctas(kv_dtype: int = KV_BF16) -> int:
    n = lib().hpc_decode_default_num_ctas(kv_dtype)
    if n <= 0:
        raise HpcError("hpc_decode_default_num_ctas", detail="device query failed")
    return n


def suggest_num_ctas(seq_lens, num_kv_heads: int, kv_dtype: int = KV_BF16, min_chunks_per_cta: int = 2,
                     q_len: int = 1) -> int:
    """hpc_decode_suggest_num_ctas on host lengths (a CPU int32 tensor or array)."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens.cpu().numpy() if isinstance(seq_lens, torch.Tensor) else seq_lens,
                              dtype=np.int32)
    n = lib().hpc_decode_suggest_num_ctas(ctypes.c_void_p(sl.ctypes.data), int(sl.shape[0]), num_kv_heads,
                                          min_chunks_per_cta, kv_dtype, q_len)
    if n <= 0:
        raise HpcError("hpc_decode_suggest_num_ctas", detail="bad arguments or device query failed")
    return n


class Plan:
    """A task map in caller-owned device memory (``buf``) plus its host header."""

    def __init__(self, batch: int, num_kv_heads: int, num_ctas: int, device):
        nbytes = lib().hpc_decode_plan_bytes(batch, num_kv_heads, num_ctas)
        if nbytes == 0:
            raise HpcError("hpc_decode_plan_bytes", detail="sizes outside the supported limits")
        self.buf = torch.empty(nbytes // 4, dtype=torch.int32, device=device)
        self.struct = PlanStruct(self.buf.data_ptr(), nbytes, 0, 0, 0, 0, 0, 0)
        self.capacity_ctas = num_ctas
        self.split_capacity = int(lib().hpc_decode_split_capacity(batch, num_kv_heads, num_ctas))

    @property
    def num_ctas(self):
        return self.struct.num_ctas

    @property
    def mode(self):
        return self.struct.mode

    def ref(self):
        return ctypes.byref(self.struct)


def hpc_decode_plan(seq_lens: torch.Tensor, num_kv_heads: int, num_ctas: int | None = None,
                    min_chunks_per_cta: int = 2, plan: Plan | None = None, stream=None) -> Plan:
    """Load-balanced task map from device-side lengths (one launch, no host sync)."""
    _cuda_i32(seq_lens, "seq_lens")
    B = seq_lens.numel()
    if num_ctas is None:
        num_ctas = default_num_ctas(KV_BF16)
    if plan is None:
        plan = Plan(B, num_kv_heads, num_ctas, seq_lens.device)
    rc = lib().hpc_decode_plan(_ptr(seq_lens), B, num_kv_heads, num_ctas, min_chunks_per_cta,
                               plan.ref(), _stream(stream))
    _check("hpc_decode_plan", rc)
    plan.split_capacity = int(lib().hpc_decode_split_capacity(B, num_kv_heads, num_ctas))
    return plan


def hpc_decode_plan_static(seq_lens: torch.Tensor, num_kv_heads: int, num_splits: int = 16,
                           plan: Plan | None = None, stream=None) -> Plan:
    """Static split-KV task map with a fixed split count (the comparison schedule)."""
    _cuda_i32(seq_lens, "seq_lens")
    B = seq_lens.numel()
    C = num_kv_heads * B * num_splits
    if plan is None:
        plan = Plan(B, num_kv_heads, C, seq_lens.device)
    rc = lib().hpc_decode_plan_static(_ptr(seq_lens), B, num_kv_heads, num_splits, plan.ref(),
                                      _stream(stream))
    _check("hpc_decode_plan_static", rc)
    plan.split_capacity = int(lib().hpc_decode_split_capacity(B, num_kv_heads, C))
    return plan


def split_buffers(plan: Plan, device=None, q_len: int = 1):
    """Allocate split_o [capacity, 8, 128] and split_lse [capacity, 8] (float32);
    with q_len > 1, [capacity, q_len, 8, 128] and [capacity, q_len, 8]."""
    device = device or plan.buf.device
    cap = plan.split_capacity
    rows = (cap, GROUP) if q_len == 1 else (cap, q_len, GROUP)
    return (torch.empty(rows + (HEAD_DIM,), dtype=torch.float32, device=device),
            torch.empty(rows, dtype=torch.float32, device=device))


def hpc_decode_attn(q, k_cache, v_cache, page_table, seq_lens, plan: Plan, split_o, split_lse,
                    k_scale=None, v_scale=None, num_pages: int | None = None, stream=None,
                    q_scale=None, engine: int | None = None, early_kv: bool = False):
    """Persistent attention over the task map; writes split_o / split_lse.
    A float8_e4m3fn q with its q_scale [B, Hq] goes to hpc_decode_attn_q8; a
    bf16 q of shape [B, q_len, Hq, 128] (several new tokens per request, causal)
    goes to hpc_decode_attn_multi. A given ``engine`` (ENGINE_AUTO, ENGINE_MMA_SYNC
    or ENGINE_TCGEN05) goes to hpc_decode_attn_multi_engine for a bf16 q of any
    q_len (hpc_decode_attn_ex for an e4m3 q). ``early_kv`` goes
    to hpc_decode_attn_ex with HPC_ATTN_EARLY_KV: the kernel gathers the KV of
    chunks without a new token before it waits for the previous kernel (the
    caller's contract is in the header)."""
    kvd = kv_dtype_of(k_cache)
    q_len = q.shape[1] if q.dim() == 4 else 1
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    Hkv = k_cache.shape[2]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (split_o, "split_o"),
                 (split_lse, "split_lse")):
        if not (t.is_cuda and t.is_contiguous()):
            raise HpcError(n, detail="must be a contiguous CUDA tensor")
    _cuda_i32(page_table, "page_table")
    _cuda_i32(seq_lens, "seq_lens")
    need = plan.split_capacity * q_len * GROUP
    if split_o.numel() < need * HEAD_DIM or split_lse.numel() < need:
        raise HpcError("split buffers", detail=f"need {plan.split_capacity} x {q_len} x 8 rows")
    npages = int(num_pages if num_pages is not None else k_cache.shape[0])
    q8 = q.dtype in (torch.float8_e4m3fn, torch.uint8)
    if q8 and q_scale is None:
        raise HpcError("hpc_decode_attn_q8", detail="an e4m3 q needs q_scale")
    if early_kv or (q8 and engine is not None):
        rc = lib().hpc_decode_attn_ex(
            _ptr(q), _ptr(q_scale), q_len, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kvd,
            npages, _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens), B, Hq, Hkv, D,
            int(k_cache.shape[1]), plan.ref(), _ptr(split_o), _ptr(split_lse),
            ENGINE_AUTO if engine is None else int(engine), ATTN_EARLY_KV if early_kv else 0, _stream(stream))
        _check("hpc_decode_attn_ex", rc)
        return
    if q8:
        rc = lib().hpc_decode_attn_q8(
            _ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), npages,
            _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens), B, Hq, Hkv, D,
            int(k_cache.shape[1]), plan.ref(), _ptr(split_o), _ptr(split_lse), _stream(stream))
        _check("hpc_decode_attn_q8", rc)
        return
    if engine is not None:  # also for one new token ([B, Hq, 128] is [B, 1, Hq, 128])
        rc = lib().hpc_decode_attn_multi_engine(
            _ptr(q), q_len, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kvd, npages,
            _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens), B, Hq, Hkv, D, int(k_cache.shape[1]),
            plan.ref(), _ptr(split_o), _ptr(split_lse), int(engine), _stream(stream))
        _check("hpc_decode_attn_multi_engine", rc)
        return
    if q.dim() == 4:
        rc = lib().hpc_decode_attn_multi(
            _ptr(q), q_len, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kvd, npages,
            _ptr(page_table), int(page_table.shape[1]), _ptr(seq_lens), B, Hq, Hkv, D, int(k_cache.shape[1]),
            plan.ref(), _ptr(split_o), _ptr(split_lse), _stream(stream))
        _check("hpc_decode_attn_multi", rc)
        return
    rc = lib().hpc_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kvd, npages, _ptr(page_table),
        int(page_table.shape[1]), _ptr(seq_lens), B, Hq, Hkv, D, int(k_cache.shape[1]), plan.ref(),
        _ptr(split_o), _ptr(split_lse), _stream(stream))
    _check("hpc_decode_attn", rc)


def hpc_decode_combine(plan: Plan, split_o, split_lse, out, out_lse=None, num_kv_heads=None,
                       stream=None):
    """LSE-weighted merge of the partials into out (bf16) and out_lse (float32).
    A 4-D out [B, q_len, Hq, 128] merges the partials of hpc_decode_attn_multi."""
    B, Hq, D = out.shape[0], out.shape[-2], out.shape[-1]
    Hkv = num_kv_heads if num_kv_heads is not None else Hq // GROUP
    if out.dim() == 4:
        rc = lib().hpc_decode_combine_multi(plan.ref(), int(out.shape[1]), _ptr(split_o), _ptr(split_lse),
                                            _ptr(out), _ptr(out_lse), B, Hq, Hkv, D, _stream(stream))
        _check("hpc_decode_combine_multi", rc)
        return
    rc = lib().hpc_decode_combine(plan.ref(), _ptr(split_o), _ptr(split_lse), _ptr(out),
                                  _ptr(out_lse), B, Hq, Hkv, D, _stream(stream))
    _check("hpc_decode_combine", rc)


def decode(q, k_cache, v_cache, page_table, seq_lens, k_scale=None, v_scale=None,
           num_ctas: int | None = None, min_chunks_per_cta: int = 2, static_splits: int | None = None,
           stream=None, q_scale=None):
    """plan -> attn -> combine with freshly allocated buffers. Returns (out, lse, plan)."""
    Hkv = k_cache.shape[2]
    if static_splits:
        plan = hpc_decode_plan_static(seq_lens, Hkv, static_splits, stream=stream)
    else:
        if num_ctas is None:
            num_ctas = default_num_ctas(kv_dtype_of(k_cache))
        plan = hpc_decode_plan(seq_lens, Hkv, num_ctas, min_chunks_per_cta, stream=stream)
    so, sl = split_buffers(plan, q_len=q.shape[1] if q.dim() == 4 else 1)
    hpc_decode_attn(q, k_cache, v_cache, page_table, seq_lens, plan, so, sl, k_scale, v_scale,
                    stream=stream, q_scale=q_scale)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    hpc_decode_combine(plan, so, sl, out, lse, Hkv, stream=stream)
    return out, lse, plan


def hpc_decode_read_error(plan: Plan) -> int:
    """Synchronise and read the task map's device error word (HPC_DEVERR_* bits)."""
    w = ctypes.c_int(0)
    rc = lib().hpc_decode_read_error(plan.ref(), ctypes.byref(w))
    if rc not in (0, 5):
        _check("hpc_decode_read_error", rc)
    return int(w.value)


def step_workspace_bytes(batch, num_q_heads, num_kv_heads, page_table_stride, num_ctas) -> int:
    return int(lib().hpc_decode_step_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                      page_table_stride, num_ctas))


def hpc_decode_step_host(h_q, h_seq_lens, h_page_table, k_cache, v_cache, workspace, h_out,
                         h_out_lse=None, k_scale=None, v_scale=None, num_ctas=None,
                         min_chunks_per_cta: int = 2, num_pages=None, stream=None):
    """One step from host tensors (pinned CPU): H2D copies, plan, attn, combine, D2H.
    Asynchronous on ``stream``; synchronise before reading h_out."""
    B, Hq, D = h_q.shape
    Hkv = k_cache.shape[2]
    if num_ctas is None:
        num_ctas = default_num_ctas(kv_dtype_of(k_cache))
    rc = lib().hpc_decode_step_host(
        _ptr(h_q), _ptr(h_seq_lens), _ptr(h_page_table), int(h_page_table.shape[1]),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype_of(k_cache),
        int(num_pages if num_pages is not None else k_cache.shape[0]), B, Hq, Hkv, D,
        int(k_cache.shape[1]), num_ctas, min_chunks_per_cta, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(h_out), _ptr(h_out_lse), _stream(stream))
    _check("hpc_decode_step_host", rc)


class StepGraph:
    """hpc_decode_step_host captured once as a CUDA graph (hpc_decode_step_graph_*).
    The tensors given here are fixed: refill the pinned host inputs in place,
    call launch(), synchronise the stream, then read h_out / h_out_lse."""

    def __init__(self, h_q, h_seq_lens, h_page_table, k_cache, v_cache, workspace, h_out, h_out_lse=None,
                 k_scale=None, v_scale=None, num_ctas=None, min_chunks_per_cta: int = 2, num_pages=None):
        B, Hq, D = h_q.shape
        Hkv = k_cache.shape[2]
        if num_ctas is None:
            num_ctas = default_num_ctas(kv_dtype_of(k_cache))
        # keep every tensor the graph points into alive as long as the graph
        self._keep = (h_q, h_seq_lens, h_page_table, k_cache, v_cache, workspace, h_out, h_out_lse, k_scale,
                      v_scale)
        handle = _vp()
        rc = lib().hpc_decode_step_graph_create(
            _ptr(h_q), _ptr(h_seq_lens), _ptr(h_page_table), int(h_page_table.shape[1]),
            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype_of(k_cache),
            int(num_pages if num_pages is not None else k_cache.shape[0]), B, Hq, Hkv, D,
            int(k_cache.shape[1]), num_ctas, min_chunks_per_cta, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(h_out), _ptr(h_out_lse), ctypes.byref(handle))
        _check("hpc_decode_step_graph_create", rc)
        self._handle = handle

    def launch(self, stream=None):
        if not self._handle:
            raise HpcError("hpc_decode_step_graph_launch", detail="the graph was closed")
        _check("hpc_decode_step_graph_launch", lib().hpc_decode_step_graph_launch(self._handle, _stream(stream)))

    def close(self):
        if self._handle:
            rc = lib().hpc_decode_step_graph_destroy(self._handle)
            self._handle = _vp()
            _check("hpc_decode_step_graph_destroy", rc)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def hpc_rope_norm(qkv, positions, cos_sin, q_weight, k_weight, slot_mapping, q_out, k_cache, v_cache,
                  q_scale=None, k_scale=None, v_scale=None, eps: float = 1e-6, num_kv_heads=None,
                  num_pages=None, error_word=None, stream=None):
    """Fused prologue: QK-norm + rotary embedding on Q and K, K/V into the cache
    slots, Q to q_out (bf16, or e4m3 codes with q_scale [T, Hq])."""
    T, H3, D = qkv.shape
    Hkv = num_kv_heads if num_kv_heads is not None else k_cache.shape[2]
    Hq = H3 - 2 * Hkv
    rc = lib().hpc_rope_norm(
        _ptr(qkv), _ptr(positions), _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(q_weight), _ptr(k_weight),
        float(eps), _ptr(slot_mapping), T, Hq, Hkv, D, int(k_cache.shape[1]), _ptr(q_out), _ptr(q_scale),
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), kv_dtype_of(k_cache),
        int(num_pages if num_pages is not None else k_cache.shape[0]), _ptr(error_word), _stream(stream))
    _check("hpc_rope_norm", rc)
