"""Helpers for the GPU parity tests: run the CUDA path through the binding and
compare it with the float64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from load_balanced_paged_02_gb300 import binding as hb
from load_balanced_paged_02_gb300 import workloads as wl

BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP8_MAX_ABS = 6e-2
LSE_ABS = 1e-3


def run(case, num_ctas=None, min_chunks=2, static_splits=None, plan=None, engine=None, early_kv=False):
    """plan -> attn -> combine on the case's device. Returns a dict of tensors."""
    Hkv = case["k_cache"].shape[2]
    if plan is None:
        if static_splits:
            plan = hb.hpc_decode_plan_static(case["seq_lens"], Hkv, static_splits)
        else:
            if num_ctas is None:
                num_ctas = hb.default_num_ctas(hb.kv_dtype_of(case["k_cache"]))
            plan = hb.hpc_decode_plan(case["seq_lens"], Hkv, num_ctas, min_chunks)
    q_len = case["q"].shape[1] if case["q"].dim() == 4 else 1
    so, sl = hb.split_buffers(plan, q_len=q_len)
    so.fill_(float("nan"))
    sl.fill_(float("nan"))
    hb.hpc_decode_attn(case["q"], case["k_cache"], case["v_cache"], case["page_table"],
                       case["seq_lens"], plan, so, sl, case["k_scale"], case["v_scale"],
                       num_pages=case["num_pages"], q_scale=case.get("q_scale"), engine=engine,
                       early_kv=early_kv)
    out = torch.full(case["q"].shape, float("nan"), dtype=torch.bfloat16, device=case["q"].device)
    lse = torch.full(case["q"].shape[:-1], float("nan"), dtype=torch.float32, device=case["q"].device)
    hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
    torch.cuda.synchronize()
    return dict(plan=plan, split_o=so, split_lse=sl, out=out, lse=lse)


def tolerances(case):
    fp8 = case["k_cache"].dtype != torch.bfloat16
    return (FP8_MAX_ABS, None) if fp8 else (BF16_MAX_ABS, BF16_MEAN_ABS)


def assert_close(got_o, got_lse, ref_o, ref_lse, case, what=""):
    """Element-wise output and LSE bounds (max abs, mean abs, LSE abs)."""
    max_abs, mean_abs = tolerances(case)
    got_o = np.asarray(got_o, dtype=np.float64).reshape(ref_o.shape)
    got_lse = np.asarray(got_lse, dtype=np.float64).reshape(ref_lse.shape)
    assert np.all(np.isfinite(got_o)), f"{what}: non-finite outputs"
    err = np.abs(got_o - ref_o)
    assert err.max() <= max_abs, f"{what}: max abs {err.max():.3g} > {max_abs}"
    if mean_abs is not None:
        assert err.mean() <= mean_abs, f"{what}: mean abs {err.mean():.3g} > {mean_abs}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_lse)), f"{what}: -inf LSE pattern differs"
    if fin.any():
        lerr = np.abs(got_lse[fin] - ref_lse[fin]).max()
        assert lerr <= LSE_ABS, f"{what}: LSE abs {lerr:.3g} > {LSE_ABS}"
    return err


def check_plan_exact(res, case, num_ctas=None, min_chunks=2, static_splits=None):
    sl = case["seq_lens"].cpu().numpy()
    Hkv = case["k_cache"].shape[2]
    if static_splits:
        ref = oracle.plan_static(sl, Hkv, static_splits)
    else:
        ref = oracle.plan(sl, Hkv, res["plan"].num_ctas, min_chunks)
    got = res["plan"].buf.cpu().numpy()
    assert got.shape == ref.shape and np.array_equal(got, ref), "task map differs from the oracle"
    return ref


def check_full(case, res, check_splits=True, host=None, rows=None, what=""):
    """Compare every output row (and every split partial) with the oracle.

    ``host`` (a host copy of the case) and ``rows`` (the oracle's full-sequence
    rows of it) may be given when several runs share one case. Returns the
    largest and mean absolute output errors and the largest LSE error."""
    if host is None:
        host = wl.to_numpy_case(case)
    shape = host["q"].shape[:-1]  # [B, Hq] or [B, q_len, Hq]
    ro, rl = oracle.attn_rows(host) if rows is None else rows
    tag = f"{what} " if what else ""
    err = assert_close(res["out"].float().cpu().numpy(), res["lse"].cpu().numpy(), ro.reshape(shape + (128,)),
                       rl.reshape(shape), case, tag + "output")
    fin = np.isfinite(rl)
    lerr = float(np.abs(res["lse"].cpu().numpy().reshape(-1)[fin] - rl[fin]).max()) if fin.any() else 0.0
    if check_splits:
        pb = res["plan"].buf.cpu().numpy()
        so, sl = oracle.attn_splits(pb, host)
        n = so.shape[0]
        assert_close(res["split_o"][:n].cpu().numpy(), res["split_lse"][:n].cpu().numpy(), so, sl,
                     case, tag + "split partials")
    return float(err.max()), float(err.mean()), lerr


def check_split_invariants(case, res):
    """At any size: combining the GPU partials in float64 with the oracle's
    combine reproduces the GPU output, and every partial LSE is finite."""
    pb = res["plan"].buf.cpu().numpy()
    n = int(pb[3])
    so = res["split_o"][:n].double().cpu().numpy()
    sl = res["split_lse"][:n].double().cpu().numpy()
    assert np.all(np.isfinite(so))
    B, Hq = case["q"].shape[0], case["q"].shape[-2]
    q_len = case["q"].shape[1] if case["q"].dim() == 4 else None
    if q_len is None:
        assert np.all(np.isfinite(sl))
    else:
        # a new token whose visible range ends before a descriptor's chunks has an
        # empty partial there (LSE -inf, output 0); only the last q_len - 1 tokens
        # of a request can be cut off, so such partials sit at the end of a pair
        assert not np.any(np.isnan(sl)) and not np.any(np.isposinf(sl))
        assert np.all(so[np.isneginf(sl)] == 0)
    o, l = oracle.combine(pb, so, sl, B, Hq, case["k_cache"].shape[2], q_len=q_len)
    got = res["out"].float().cpu().numpy()
    # the only difference is the float32 merge and the bf16 rounding of the output
    assert np.all(np.abs(got - o) <= 2.0 ** -8 * np.abs(o) + 1e-5)
    fin = np.isfinite(l)
    assert np.abs(res["lse"].cpu().numpy()[fin] - l[fin]).max() <= 1e-4
