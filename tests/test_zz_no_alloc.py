"""The allocation-free entry point (GPU only).

hpc_decode_noalloc is for callers that cannot allocate device memory where
they run a decode step: an engine whose memory pool takes all device memory at
start-up and forbids allocations outside it, or plugin code that only receives
input and output pointers and has no allocator to reach. It keeps the task map
and split buffers in a fixed array inside the library. Calls in a row, each on
different lengths (the last one sized just under the array's limit, so that
its last split row sits near the end of the array), must match the allocating
plan -> attn -> combine path and the float64 oracle within the parity
tolerances; sizes beyond the fixed array must be refused before any work.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import _gpu
import oracle
from load_balanced_paged_02_gb300 import _build
from load_balanced_paged_02_gb300 import binding as hb
from load_balanced_paged_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ARRAY_BYTES = 8 << 20  # the library's fixed array


def _noalloc(L, case, C, m, out, lse):
    B, Hq, D = case["q"].shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.hpc_decode_noalloc(p(case["q"]), p(case["k_cache"]), p(case["v_cache"]),
                                p(case["k_scale"]), p(case["v_scale"]), hb.kv_dtype_of(case["k_cache"]),
                                case["num_pages"], p(case["page_table"]), case["page_table"].shape[1],
                                p(case["seq_lens"]), B, Hq, case["k_cache"].shape[2], D,
                                case["k_cache"].shape[1], C, m, p(out), p(lse), stream)


def _need_bytes(L, B, Hkv, C):
    """The header's size rule: the task map plus hpc_decode_split_capacity rows
    of 4128 bytes (8 x 128 + 8 float32), each part rounded up to 256 bytes."""
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    cap = L.hpc_decode_split_capacity(B, Hkv, C)
    return r(L.hpc_decode_plan_bytes(B, Hkv, C)) + r(cap * 8 * 128 * 4) + r(cap * 8 * 4)


def _largest_batch(L, Hkv, C):
    B = 1
    while _need_bytes(L, B + 1, Hkv, C) <= ARRAY_BYTES:
        B += 1
    return B


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return hb.lib()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_noalloc_matches_allocating_path_and_oracle(L, dtype):
    C = hb.default_num_ctas(hb.KV_FP8_E4M3 if dtype == "fp8" else hb.KV_BF16)
    rng = np.random.default_rng(31)
    b_max = _largest_batch(L, 8, C)
    # three different batches in a row: no call may depend on an earlier call's
    # contents of the array; the last fills it to within one request
    batches = [rng.integers(1, 9000, size=24).tolist(), rng.integers(0, 3000, size=9).tolist(),
               rng.integers(100, 3000, size=b_max).tolist()]
    max_abs = 6e-2 if dtype == "fp8" else 2e-2
    for i, lens in enumerate(batches):
        w = wl.Workload(f"noalloc{i}", len(lens), 64, 8, dtype, 40 + i, lens=lens)
        case = wl.make_case(w, device=DEV)
        if i == 2:
            # the task map's split rows reach close to the capacity the size
            # rule reserves, so the last rows written sit near the array's end
            cap = L.hpc_decode_split_capacity(len(lens), 8, C)
            splits = int(oracle.plan(np.asarray(lens, np.int32), 8, C, 2)[3])
            assert splits >= cap - C // 4, (splits, cap)
            assert _need_bytes(L, len(lens), 8, C) > ARRAY_BYTES - 64 * 1024
        ref_out, ref_lse, _ = hb.decode(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                                        case["seq_lens"], case["k_scale"], case["v_scale"], num_ctas=C,
                                        min_chunks_per_cta=2)
        out = torch.full_like(case["q"], float("nan"))
        lse = torch.full(case["q"].shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(L, case, C, 2, out, lse) == 0
        torch.cuda.synchronize()
        # against the existing (allocating) entry points
        err = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= max_abs
        if dtype == "bf16":
            assert err.mean().item() <= 2e-3
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= 1e-3
        # against the float64 oracle, every row
        host = wl.to_numpy_case(case)
        ro, rl = oracle.attn_rows(host)
        B, Hq = len(lens), 64
        _gpu.assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), ro.reshape(B, Hq, 128),
                          rl.reshape(B, Hq), case, f"allocation-free call {i}")


def test_noalloc_refuses_sizes_beyond_its_array(L):
    fake = ctypes.c_void_p(0x10000)  # refused before any pointer is used
    # 4096 requests x 8 KV heads need ~32k split rows (~135 MB), far above 8 MiB
    rc = L.hpc_decode_noalloc(fake, fake, fake, None, None, 0, 1000, fake, 8, fake, 4096, 64, 8, 128, 64,
                              152, 2, fake, None, None)
    assert rc == 3
    # one request more than fits: refused, with real buffers, and nothing written
    C = hb.default_num_ctas(hb.KV_BF16)
    B = _largest_batch(L, 8, C) + 1
    w = wl.Workload("noalloc_over", B, 64, 8, "bf16", 45, lens=[64] * B)
    case = wl.make_case(w, device=DEV)
    out = torch.full_like(case["q"], float("nan"))
    assert _noalloc(L, case, C, 2, out, None) == 3
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
