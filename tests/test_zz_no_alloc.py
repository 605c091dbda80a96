"""The allocation-free entry point against the allocating path (GPU only).

hpc_decode_noalloc is for callers that cannot allocate device memory where
they run a decode step (an engine whose pool owns all device memory, or a
plugin that only receives input and output pointers): it keeps the task map
and split buffers in a fixed array inside the library. Two calls in a row,
each on different lengths, must match plan -> attn -> combine with
caller-owned buffers within the parity tolerances; sizes beyond the fixed
array must be refused. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from load_balanced_paged_02_gb300 import _build
from load_balanced_paged_02_gb300 import binding as hb
from load_balanced_paged_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _noalloc(L, case, C, m, out, lse):
    B, Hq, D = case["q"].shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.hpc_decode_noalloc(p(case["q"]), p(case["k_cache"]), p(case["v_cache"]),
                                p(case["k_scale"]), p(case["v_scale"]), hb.kv_dtype_of(case["k_cache"]),
                                case["num_pages"], p(case["page_table"]), case["page_table"].shape[1],
                                p(case["seq_lens"]), B, Hq, case["k_cache"].shape[2], D,
                                case["k_cache"].shape[1], C, m, p(out), p(lse), stream)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_noalloc_matches_allocating_path_twice(dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    L = hb.lib()
    C = hb.default_num_ctas(hb.KV_FP8_E4M3 if dtype == "fp8" else hb.KV_BF16)
    rng = np.random.default_rng(31)
    # two different batches: the second call must not see the first call's state
    batches = [rng.integers(1, 9000, size=24).tolist(), rng.integers(0, 3000, size=9).tolist()]
    max_abs = 6e-2 if dtype == "fp8" else 2e-2
    for i, lens in enumerate(batches):
        w = wl.Workload(f"noalloc{i}", len(lens), 64, 8, dtype, 40 + i, lens=lens)
        case = wl.make_case(w, device=DEV)
        ref_out, ref_lse, _ = hb.decode(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                                        case["seq_lens"], case["k_scale"], case["v_scale"], num_ctas=C,
                                        min_chunks_per_cta=2)
        out = torch.full_like(case["q"], float("nan"))
        lse = torch.full(case["q"].shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(L, case, C, 2, out, lse) == 0
        torch.cuda.synchronize()
        err = (out.float() - ref_out.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= max_abs
        if dtype == "bf16":
            assert err.mean().item() <= 2e-3
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= 1e-3


def test_noalloc_refuses_sizes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    L = hb.lib()
    fake = ctypes.c_void_p(0x10000)  # refused before any pointer is used
    # 4096 requests x 8 KV heads need ~32k split rows (~135 MB), far above 8 MiB
    rc = L.hpc_decode_noalloc(fake, fake, fake, None, None, 0, 1000, fake, 8, fake, 4096, 64, 8, 128, 64,
                              152, 2, fake, None, None)
    assert rc == 3
