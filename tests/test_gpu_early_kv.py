"""Attention that gathers KV before it waits for the kernel before it
(HPC_ATTN_EARLY_KV; "SGLang Low-Latency Mode: Kernels and Runtime", section
"Low-Latency-Specific Optimizations", item 1) — GPU only.

The early copies are the same copies the producer would issue later, so every
partial, LSE and output must be bit-identical to the call without the flag,
for every kernel (one-token, warp-level multi-token, tcgen05, e4m3 query).
The chained test runs the layer as a caller would: plan, then the fused
prologue writing each request's new tokens into a cache whose new-token slots
hold large poison values, then early attention and combine, all queued on one
stream with no synchronisation; the result must match the float64 oracle run
on the cache the prologue leaves (the oracle side uses only its own prologue).
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

# chunk boundaries, one-chunk and sub-chunk requests, long runs that fill the
# ring, and requests shorter than the new-token count
LENS = [1, 63, 64, 65, 130, 700, 4096, 5000, 129, 3, 2048, 9000, 7, 640]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hb.lib()


def _same_bits(a, b, what):
    a, b = a.contiguous(), b.contiguous()
    assert a.shape == b.shape, what
    ia = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
    ib = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
    assert torch.equal(ia, ib), f"{what}: {(ia != ib).sum().item()} elements differ"


CASES = [
    # (kv dtype, q_len, engine, e4m3 query)
    ("bf16", 1, None, False),
    ("bf16", 1, hb.ENGINE_TCGEN05, False),
    ("fp8", 1, None, False),
    ("fp8", 1, None, True),
    ("bf16", 2, hb.ENGINE_MMA_SYNC, False),
    ("bf16", 5, hb.ENGINE_MMA_SYNC, False),
    ("bf16", 5, hb.ENGINE_TCGEN05, False),
    ("bf16", 8, hb.ENGINE_TCGEN05, False),
    ("fp8", 2, hb.ENGINE_MMA_SYNC, False),
    ("fp8", 6, hb.ENGINE_MMA_SYNC, False),
    ("fp8", 3, hb.ENGINE_TCGEN05, False),
    ("fp8", 8, hb.ENGINE_TCGEN05, False),
]


@pytest.mark.parametrize("num_ctas", [24, None])
@pytest.mark.parametrize("kv,q_len,engine,q8", CASES)
def test_bit_identical_to_plain_call(kv, q_len, engine, q8, num_ctas):
    w = wl.Workload("early", len(LENS), 64, 8, kv, 41, lens=LENS, q_len=q_len, q_dtype="fp8" if q8 else "bf16")
    case = wl.make_case(w, device=DEV)
    plain = _gpu.run(case, num_ctas=num_ctas, engine=engine)
    early = _gpu.run(case, plan=plain["plan"], engine=engine, early_kv=True)
    assert hb.hpc_decode_read_error(plain["plan"]) == 0
    for k in ("split_o", "split_lse", "out", "lse"):
        _same_bits(early[k], plain[k], k)


@pytest.mark.parametrize("kv,q_len,engine", [("bf16", 1, None), ("fp8", 1, None), ("bf16", 4, hb.ENGINE_TCGEN05),
                                             ("fp8", 6, hb.ENGINE_TCGEN05), ("bf16", 3, hb.ENGINE_MMA_SYNC)])
def test_early_path_matches_oracle(kv, q_len, engine):
    w = wl.Workload("early", len(LENS), 64, 8, kv, 43, lens=LENS, q_len=q_len)
    case = wl.make_case(w, device=DEV)
    res = _gpu.run(case, num_ctas=24, engine=engine, early_kv=True)
    _gpu.check_full(case, res)


def _round_bf16(x):
    return torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _quant_e4m3(x):
    s = np.abs(x).max(axis=-1) / 448.0
    s[s == 0] = 1.0
    c = torch.from_numpy(x / s[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return c, s.astype(np.float32)


@pytest.mark.parametrize("kv,q_len,engine", [("bf16", 1, None), ("fp8", 1, None), ("bf16", 2, hb.ENGINE_MMA_SYNC),
                                             ("bf16", 6, hb.ENGINE_TCGEN05), ("fp8", 4, hb.ENGINE_TCGEN05)])
def test_chain_plan_prologue_early_attention(kv, q_len, engine):
    lens = [8, 64, 65, 127, 640, 3000, 5000, 129, 4096, 200, 70, 1500]
    B, Hq, Hkv = len(lens), 64, 8
    fp8 = kv == "fp8"
    q8 = fp8 and q_len == 1  # the e4m3 query goes with the one-token e4m3 kernel
    w = wl.Workload("chain", B, Hq, Hkv, kv, 47, lens=lens, q_len=q_len)
    case = wl.make_case(w, device=DEV)
    pt = case["page_table"].cpu().numpy()
    pos = np.array([L - q_len + i for L in lens for i in range(q_len)], dtype=np.int32)
    req = np.repeat(np.arange(B), q_len)
    slots = (pt[req, pos // 64] * 64 + pos % 64).astype(np.int32)
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=48, device=DEV, max_pos=8192, slots=slots)

    # poison the slots the prologue is about to write
    pg = torch.from_numpy((slots // 64).astype(np.int64)).to(DEV)
    off = torch.from_numpy((slots % 64).astype(np.int64)).to(DEV)
    if fp8:
        case["k_cache"].view(torch.uint8)[pg, off] = 0x7E  # 448
        case["v_cache"].view(torch.uint8)[pg, off] = 0x7E
        case["k_scale"][pg, :, off] = 100.0
        case["v_scale"][pg, :, off] = 100.0
    else:
        case["k_cache"][pg, off] = 64.0
        case["v_cache"][pg, off] = 64.0
    host = wl.to_numpy_case(case)  # poisoned cache: the oracle overwrites the same slots below
    torch.cuda.synchronize()

    T = B * q_len
    q_out = torch.empty((T, Hq, 128), dtype=torch.float8_e4m3fn if q8 else torch.bfloat16, device=DEV)
    q_sc = torch.empty((T, Hq), dtype=torch.float32, device=DEV) if q8 else None
    plan = hb.hpc_decode_plan(case["seq_lens"], Hkv, 40, 2)
    hb.hpc_rope_norm(pc["qkv"], pc["positions"], pc["cos_sin"], pc["q_weight"], pc["k_weight"], pc["slots"],
                     q_out, case["k_cache"], case["v_cache"], q_scale=q_sc, k_scale=case["k_scale"],
                     v_scale=case["v_scale"], eps=pc["eps"], num_kv_heads=Hkv)
    q_in = q_out if q_len == 1 else q_out.view(B, q_len, Hq, 128)
    so, sl = hb.split_buffers(plan, q_len=q_len)
    hb.hpc_decode_attn(q_in, case["k_cache"], case["v_cache"], case["page_table"], case["seq_lens"], plan, so, sl,
                       case["k_scale"], case["v_scale"], num_pages=case["num_pages"], q_scale=q_sc,
                       engine=engine, early_kv=True)
    out = torch.empty(q_in.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(q_in.shape[:-1], dtype=torch.float32, device=DEV)
    hb.hpc_decode_combine(plan, so, sl, out, lse, Hkv)
    torch.cuda.synchronize()
    assert hb.hpc_decode_read_error(plan) == 0

    bits = pc["qkv"].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    rq, rk, rv = oracle.rope_norm(bits, pos, pc["cos_sin"].cpu().numpy(), pc["q_weight"].cpu().numpy(),
                                  pc["k_weight"].cpu().numpy(), pc["eps"], Hq, Hkv)
    if fp8:
        kc, ksc = _quant_e4m3(rk)
        vc, vsc = _quant_e4m3(rv)
    else:
        kc, vc = _round_bf16(rk), _round_bf16(rv)
    for t, s in enumerate(slots):
        p_, o_ = s // 64, s % 64
        host["k_cache"][p_, o_], host["v_cache"][p_, o_] = kc[t], vc[t]
        if fp8:
            host["k_scale"][p_, :, o_], host["v_scale"][p_, :, o_] = ksc[t], vsc[t]
    if q8:
        host["q"], host["q_scale"] = _quant_e4m3(rq)
    else:
        qb = _round_bf16(rq)
        host["q"] = qb if q_len == 1 else qb.reshape(B, q_len, Hq, 128)
        host.pop("q_scale", None)
    ro, rl = oracle.attn_rows(host)
    shape = q_in.shape[:-1]
    _gpu.assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), ro.reshape(shape + (128,)), rl.reshape(shape),
                      case, "plan -> prologue -> early attention -> combine")
