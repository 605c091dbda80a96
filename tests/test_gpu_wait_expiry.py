"""The attention kernel's timeout path, taken on purpose (GPU only).

Every wait inside the attention kernels is bounded; when one runs out the CTA
records HPC_DEVERR_WAIT_TIMEOUT in the task map's error word, waits for its
own copies in flight and returns, so the device stays usable. The flag
HPC_ATTN_TEST_WAIT_EXPIRY makes the consumer warps of the one-token kernel
wait, with a 1 ms limit, on a barrier that nothing completes. Nothing faults,
traps or hangs: the test checks that the call returns, that the error word
says what happened, that no partial was written, and that the next ordinary
call on the same stream is exact against the oracle.
"""
import ctypes
import time

import pytest
import torch

import _gpu
from load_balanced_paged_02_gb300 import binding as hb
from load_balanced_paged_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
WAIT_TIMEOUT = 8  # HPC_DEVERR_WAIT_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hb.lib()


def _attn_ex(case, plan, so, sl, flags, engine=hb.ENGINE_AUTO):
    B, Hq, D = case["q"].shape
    p = hb._ptr
    return hb.lib().hpc_decode_attn_ex(
        p(case["q"]), None, 1, p(case["k_cache"]), p(case["v_cache"]), p(case["k_scale"]), p(case["v_scale"]),
        hb.kv_dtype_of(case["k_cache"]), case["num_pages"], p(case["page_table"]), case["page_table"].shape[1],
        p(case["seq_lens"]), B, Hq, case["k_cache"].shape[2], D, case["k_cache"].shape[1], plan.ref(), p(so),
        p(sl), engine, flags, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("num_ctas", [1, 152, 400])
def test_wait_runs_out_then_next_call_is_exact(dtype, num_ctas):
    """One CTA with a long list (its producer is blocked on a full ring when
    the consumers leave), one CTA per SM (most producers finish their short
    lists first and drain at the end), and the shallow instance's two CTAs
    per SM."""
    lens = [1000, 64, 4097, 300, 0, 129, 2000, 65, 7, 900]
    w = wl.Workload("expiry", len(lens), 16, 2, dtype, 70 + num_ctas, lens=lens)
    case = wl.make_case(w, device=DEV)
    plan = hb.hpc_decode_plan(case["seq_lens"], 2, num_ctas, 1)
    so, sl = hb.split_buffers(plan)
    so.fill_(float("nan"))
    sl.fill_(float("nan"))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _attn_ex(case, plan, so, sl, hb.ATTN_TEST_WAIT_EXPIRY) == 0
    err = hb.hpc_decode_read_error(plan)  # synchronises
    elapsed = time.perf_counter() - t0
    assert err == WAIT_TIMEOUT, f"error word {err:#x}"
    assert torch.isnan(so).all() and torch.isnan(sl).all(), "a partial was written after the timeout"
    # well under the kernels' ordinary 2 s limit: the 1 ms test wait ran out
    assert elapsed < 1.5, f"{elapsed:.2f} s"
    # the device is usable and the next step on the same buffers is exact
    hb.hpc_decode_plan(case["seq_lens"], 2, num_ctas, 1, plan=plan)
    assert _attn_ex(case, plan, so, sl, 0) == 0
    out = torch.empty_like(case["q"])
    lse = torch.empty(case["q"].shape[:2], dtype=torch.float32, device=DEV)
    hb.hpc_decode_combine(plan, so, sl, out, lse, 2)
    torch.cuda.synchronize()
    assert hb.hpc_decode_read_error(plan) == 0
    _gpu.check_full(case, dict(plan=plan, split_o=so, split_lse=sl, out=out, lse=lse))


def test_flag_refused_outside_the_one_token_kernel():
    lens = [100, 200]
    case = wl.make_case(wl.Workload("expiry", 2, 8, 1, "bf16", 77, lens=lens), device=DEV)
    plan = hb.hpc_decode_plan(case["seq_lens"], 1, 4, 1)
    so, sl = hb.split_buffers(plan)
    assert _attn_ex(case, plan, so, sl, hb.ATTN_TEST_WAIT_EXPIRY, engine=hb.ENGINE_TCGEN05) == 2
    torch.cuda.synchronize()
    assert hb.hpc_decode_read_error(plan) == 0
