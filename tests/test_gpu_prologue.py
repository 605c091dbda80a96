"""Fused attention prologue (HpcRopeNorm) against the float64 oracle (GPU only).

bf16 outputs: within one bf16 rounding of the oracle value (plus float32
arithmetic). e4m3 outputs are integers decided by floating point, so they are
checked for validity: the scale is amax/448 of the oracle's row (relative
1e-4), and each code is a nearest e4m3 value of oracle/scale (at most half a
grid step away, with float32 slack); almost all codes equal the oracle's own
rounding. The chained decode test runs prologue -> attention on both sides:
the oracle side only uses the oracle's own prologue output.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hb.lib()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _oracle(pc):
    return oracle.rope_norm(_bits(pc["qkv"]), pc["positions"].cpu().numpy(), pc["cos_sin"].cpu().numpy(),
                            pc["q_weight"].cpu().numpy(), pc["k_weight"].cpu().numpy(), pc["eps"],
                            pc["num_q_heads"], pc["num_kv_heads"])


def _e4m3_grid_step(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -9)))
    return 2.0 ** (np.maximum(e, -6) - 3)


def check_e4m3_rows(codes_u8, scales, ref, what):
    """codes [..., 128] uint8, scales [...] float32, ref [..., 128] float64."""
    ref_scale = np.abs(ref).max(axis=-1) / 448.0
    ref_scale[ref_scale == 0] = 1.0
    assert np.allclose(scales, ref_scale, rtol=1e-4, atol=0), f"{what}: scales"
    val = torch.from_numpy(codes_u8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = ref / scales.astype(np.float64)[..., None]
    # float32 norm/rotation error is relative to the row's magnitude (about 4 ulp
    # of the row max = 448 in code units), not to each element
    slack = 2e-5 * np.abs(v) + 4 * 2.0 ** -23 * 448
    excess = np.abs(val - v) - (0.5 * _e4m3_grid_step(v) + slack)
    bad = excess > 0
    assert not bad.any(), (f"{what}: {int(bad.sum())} codes not a nearest value; worst excess "
                           f"{excess.max():.3g} at v={v[np.unravel_index(excess.argmax(), v.shape)]:.6g}")
    own = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.mean(own != val) < 1e-3, f"{what}: too many codes differ from the oracle's rounding"


def run_prologue(pc, q_fp8, kv_fp8, num_pages, err=None):
    T = pc["qkv"].shape[0]
    Hq, Hkv = pc["num_q_heads"], pc["num_kv_heads"]
    kv_dt = torch.float8_e4m3fn if kv_fp8 else torch.bfloat16
    k = torch.full((num_pages, 64, Hkv, 128), 3.0, device=DEV).to(kv_dt)
    v = torch.full((num_pages, 64, Hkv, 128), 3.0, device=DEV).to(kv_dt)
    ks = torch.full((num_pages, Hkv, 64), -7.0, device=DEV) if kv_fp8 else None
    vs = torch.full((num_pages, Hkv, 64), -7.0, device=DEV) if kv_fp8 else None
    q = torch.empty((T, Hq, 128), dtype=torch.float8_e4m3fn if q_fp8 else torch.bfloat16, device=DEV)
    qs = torch.empty((T, Hq), dtype=torch.float32, device=DEV) if q_fp8 else None
    hb.hpc_rope_norm(pc["qkv"], pc["positions"], pc["cos_sin"], pc["q_weight"], pc["k_weight"], pc["slots"],
                     q, k, v, q_scale=qs, k_scale=ks, v_scale=vs, eps=pc["eps"], num_kv_heads=Hkv,
                     error_word=err)
    torch.cuda.synchronize()
    return q, qs, k, v, ks, vs


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (64, 8)])
def test_bf16_outputs_and_slots(Hq, Hkv):
    T = 37
    rng = np.random.default_rng(0)
    pos = rng.integers(0, 8000, size=T).astype(np.int32)
    slots = rng.permutation(10 * 64)[:T].astype(np.int32)
    slots[5] = -1  # a padding token: nothing written
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=1, device=DEV, max_pos=8192, slots=slots)
    q, _, k, v, _, _ = run_prologue(pc, False, False, num_pages=10)
    rq, rk, rv = _oracle(pc)
    tol = lambda r: 2.0 ** -8 * np.abs(r) + 2e-5  # noqa: E731
    assert np.all(np.abs(q.float().cpu().numpy() - rq) <= tol(rq))
    kc, vc = k.float().cpu().numpy(), v.float().cpu().numpy()
    written = np.zeros((10 * 64,), dtype=bool)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        written[sl] = True
        assert np.all(np.abs(kc[sl // 64, sl % 64] - rk[t]) <= tol(rk[t]))
        assert np.array_equal(vc[sl // 64, sl % 64], rv[t].astype(np.float32))
    untouched = kc.reshape(640, Hkv, 128)[~written]
    assert np.all(untouched == 3.0) and np.all(vc.reshape(640, Hkv, 128)[~written] == 3.0)


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (64, 8)])
def test_e4m3_outputs(Hq, Hkv):
    T = 29
    rng = np.random.default_rng(1)
    pos = rng.integers(0, 8000, size=T).astype(np.int32)
    slots = rng.permutation(6 * 64)[:T].astype(np.int32)
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=2, device=DEV, max_pos=8192, slots=slots)
    q, qs, k, v, ks, vs = run_prologue(pc, True, True, num_pages=6)
    rq, rk, rv = _oracle(pc)
    check_e4m3_rows(q.view(torch.uint8).cpu().numpy(), qs.cpu().numpy(), rq, "q")
    kc, vc = k.view(torch.uint8).cpu().numpy(), v.view(torch.uint8).cpu().numpy()
    ksc, vsc = ks.cpu().numpy(), vs.cpu().numpy()
    for t, sl in enumerate(slots):
        pg, off = sl // 64, sl % 64
        check_e4m3_rows(kc[pg, off], ksc[pg, :, off], rk[t], f"k token {t}")
        check_e4m3_rows(vc[pg, off], vsc[pg, :, off], rv[t], f"v token {t}")


def test_many_rows_path_matches_oracle():
    """Enough rows that each warp takes eight of them (prefill-sized call)."""
    T = 1000  # 1000 x 80 rows
    rng = np.random.default_rng(9)
    pos = rng.integers(0, 4000, size=T).astype(np.int32)
    pc = wl.make_prologue_case(pos, 64, 8, seed=9, device=DEV, max_pos=4096,
                               slots=np.arange(T, dtype=np.int32))
    q, qs, k, v, ks, vs = run_prologue(pc, True, True, num_pages=16)
    rq, rk, rv = _oracle(pc)
    check_e4m3_rows(q.view(torch.uint8).cpu().numpy(), qs.cpu().numpy(), rq, "q")
    kc = k.view(torch.uint8).cpu().numpy().reshape(1024, 8, 128)[:T]
    vc = v.view(torch.uint8).cpu().numpy().reshape(1024, 8, 128)[:T]
    ksc = ks.cpu().numpy().transpose(0, 2, 1).reshape(1024, 8)[:T]
    vsc = vs.cpu().numpy().transpose(0, 2, 1).reshape(1024, 8)[:T]
    check_e4m3_rows(kc, ksc, rk, "k")
    check_e4m3_rows(vc, vsc, rv, "v")


@pytest.mark.parametrize("fp8", [False, True])
def test_large_call_instance_matches_oracle(fp8):
    """A call of at least four waves of blocks (2600 tokens x 80 rows) runs the
    prologue's 64-register instance (four blocks per SM)."""
    T = 2600
    rng = np.random.default_rng(12)
    pos = rng.integers(0, 4000, size=T).astype(np.int32)
    pc = wl.make_prologue_case(pos, 64, 8, seed=12, device=DEV, max_pos=4096,
                               slots=np.arange(T, dtype=np.int32))
    pages = (T + 63) // 64
    q, qs, k, v, ks, vs = run_prologue(pc, fp8, fp8, num_pages=pages)
    rq, rk, rv = _oracle(pc)
    if fp8:
        check_e4m3_rows(q.view(torch.uint8).cpu().numpy(), qs.cpu().numpy(), rq, "q")
        kc = k.view(torch.uint8).cpu().numpy().reshape(pages * 64, 8, 128)[:T]
        ksc = ks.cpu().numpy().transpose(0, 2, 1).reshape(pages * 64, 8)[:T]
        check_e4m3_rows(kc, ksc, rk, "k")
        vc = v.view(torch.uint8).cpu().numpy().reshape(pages * 64, 8, 128)[:T]
        vsc = vs.cpu().numpy().transpose(0, 2, 1).reshape(pages * 64, 8)[:T]
        check_e4m3_rows(vc, vsc, rv, "v")
    else:
        tol = lambda r: 2.0 ** -8 * np.abs(r) + 2e-5  # noqa: E731
        assert np.all(np.abs(q.float().cpu().numpy() - rq) <= tol(rq))
        kc = k.float().cpu().numpy().reshape(pages * 64, 8, 128)[:T]
        vc = v.float().cpu().numpy().reshape(pages * 64, 8, 128)[:T]
        assert np.all(np.abs(kc - rk) <= tol(rk))
        assert np.array_equal(vc, rv.astype(np.float32))


def _check_large(pc, q_fp8, kv_fp8, slots, pages, what):
    q, qs, k, v, ks, vs = run_prologue(pc, q_fp8, kv_fp8, num_pages=pages)
    rq, rk, rv = _oracle(pc)
    Hkv = pc["num_kv_heads"]
    tol = lambda r: 2.0 ** -8 * np.abs(r) + 2e-5  # noqa: E731
    if q_fp8:
        check_e4m3_rows(q.view(torch.uint8).cpu().numpy(), qs.cpu().numpy(), rq, f"{what} q")
    else:
        assert np.all(np.abs(q.float().cpu().numpy() - rq) <= tol(rq)), f"{what} q"
    live = slots >= 0
    sl = slots[live]
    if kv_fp8:
        kc = k.view(torch.uint8).cpu().numpy().reshape(pages * 64, Hkv, 128)
        vc = v.view(torch.uint8).cpu().numpy().reshape(pages * 64, Hkv, 128)
        ksc = ks.cpu().numpy().transpose(0, 2, 1).reshape(pages * 64, Hkv)
        vsc = vs.cpu().numpy().transpose(0, 2, 1).reshape(pages * 64, Hkv)
        check_e4m3_rows(kc[sl], ksc[sl], rk[live], f"{what} k")
        check_e4m3_rows(vc[sl], vsc[sl], rv[live], f"{what} v")
        untouched = np.ones(pages * 64, dtype=bool)
        untouched[sl] = False
        assert np.all(ksc[untouched] == -7.0) and np.all(vsc[untouched] == -7.0), f"{what}: stray writes"
    else:
        kc = k.float().cpu().numpy().reshape(pages * 64, Hkv, 128)
        vc = v.float().cpu().numpy().reshape(pages * 64, Hkv, 128)
        assert np.all(np.abs(kc[sl] - rk[live]) <= tol(rk[live])), f"{what} k"
        assert np.array_equal(vc[sl], rv[live].astype(np.float32)), f"{what} v"
        untouched = np.ones(pages * 64, dtype=bool)
        untouched[sl] = False
        assert np.all(kc[untouched] == 3.0) and np.all(vc[untouched] == 3.0), f"{what}: stray writes"


@pytest.mark.parametrize("Hq,Hkv,T", [(8, 1, 5001), (12, 3, 2500), (64, 8, 1203)])
@pytest.mark.parametrize("q_fp8,kv_fp8", [(False, False), (True, True), (False, True), (True, False)])
def test_prefill_ring_kernel_matches_oracle(Hq, Hkv, T, q_fp8, kv_fp8):
    """Prefill-sized calls (at least two ring stages per SM) run the ring-fed
    kernel: 8/1 heads (16 tokens per stage), 12/3 heads (18 rows per token, so
    a 4-row unit straddles two tokens), 64/8 heads; a partial last stage;
    padding slots (-1, nothing written) among shuffled slots; every output
    format combination."""
    rng = np.random.default_rng(T + Hq)
    pos = rng.integers(0, 4000, size=T).astype(np.int32)
    pages = (T + 63) // 64 + 2
    slots = rng.permutation(pages * 64)[:T].astype(np.int32)
    slots[::97] = -1
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=T, device=DEV, max_pos=4096, slots=slots)
    _check_large(pc, q_fp8, kv_fp8, slots, pages, f"{Hq}/{Hkv} T={T}")


def test_prefill_ring_kernel_error_bits():
    """A bad position (not rotated) and an out-of-range slot (nothing written)
    in a prefill-sized call set their error bits; the other rows are exact."""
    T, Hq, Hkv = 5000, 8, 1
    pos = (np.arange(T) % 4000).astype(np.int32)
    pos[17] = 5000
    pages = (T + 63) // 64
    slots = np.arange(T, dtype=np.int32)
    slots[33] = pages * 64 + 5
    pc = wl.make_prologue_case(pos, Hq, Hkv, seed=5, device=DEV, max_pos=4096, slots=slots)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, _, k, _, _, _ = run_prologue(pc, False, False, num_pages=pages, err=err)
    assert int(err.item()) & 32 and int(err.item()) & 4
    good = pos.copy()
    good[17] = 0  # the bad position's rows are normalised but not rotated (identity rotation at 0)
    rq, rk, _ = _oracle(dict(pc, positions=torch.from_numpy(good).to(DEV)))
    tol = lambda r: 2.0 ** -8 * np.abs(r) + 2e-5  # noqa: E731
    assert np.all(np.abs(q.float().cpu().numpy() - rq) <= tol(rq))
    kc = k.float().cpu().numpy().reshape(pages * 64, Hkv, 128)
    live = np.arange(T) != 33
    assert np.all(np.abs(kc[slots[live]] - rk[live]) <= tol(rk[live]))


def test_bad_position_sets_error_bit():
    pc = wl.make_prologue_case([3, 9000, 5], 8, 1, seed=3, device=DEV, max_pos=16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, _, _, _, _, _ = run_prologue(pc, False, False, num_pages=2, err=err)
    assert int(err.item()) & 32
    good = _oracle(dict(pc, positions=torch.tensor([3, 0, 5], dtype=torch.int32)))[0]
    # rows of valid positions are exact; the bad row is normalised but not rotated
    assert np.allclose(q[[0, 2]].float().cpu().numpy(), good[[0, 2]], rtol=2 ** -8, atol=2e-5)
    assert np.allclose(q[1].float().cpu().numpy(), good[1], rtol=2 ** -8, atol=2e-5)


def test_decode_chain_prologue_then_e4m3_attention():
    """One decode step: the prologue writes each request's newest K/V into the
    e4m3 cache and emits the e4m3 query; attention then reads both. The oracle
    runs its own prologue, rounds it the same way (torch e4m3 conversion),
    writes a host copy of the cache, and runs its attention."""
    lens = [1, 70, 640, 3000, 64, 129]
    w = wl.Workload("chain", len(lens), 64, 8, "fp8", 31, lens=lens)
    case = wl.make_case(w, device=DEV)
    slots = wl.decode_slots(case)
    pos = np.asarray(lens, dtype=np.int32) - 1
    pc = wl.make_prologue_case(pos, 64, 8, seed=32, device=DEV, max_pos=4096, slots=slots)
    q8 = torch.empty((len(lens), 64, 128), dtype=torch.float8_e4m3fn, device=DEV)
    qs = torch.empty((len(lens), 64), dtype=torch.float32, device=DEV)
    host = wl.to_numpy_case(case)  # cache before the prologue writes (oracle side)
    hb.hpc_rope_norm(pc["qkv"], pc["positions"], pc["cos_sin"], pc["q_weight"], pc["k_weight"], pc["slots"],
                     q8, case["k_cache"], case["v_cache"], q_scale=qs, k_scale=case["k_scale"],
                     v_scale=case["v_scale"], eps=pc["eps"], num_kv_heads=8)
    gpu_case = dict(case, q=q8, q_scale=qs)
    res = _gpu.run(gpu_case, num_ctas=40)

    rq, rk, rv = _oracle(pc)

    def quant(x):
        s = np.abs(x).max(axis=-1) / 448.0
        s[s == 0] = 1.0
        c = torch.from_numpy(x / s[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return c, s.astype(np.float32)

    qc, qsc = quant(rq)
    kc, ksc = quant(rk)
    vc, vsc = quant(rv)
    for b, sl in enumerate(slots):
        pg, off = sl // 64, sl % 64
        host["k_cache"][pg, off], host["v_cache"][pg, off] = kc[b], vc[b]
        host["k_scale"][pg, :, off], host["v_scale"][pg, :, off] = ksc[b], vsc[b]
    host["q"], host["q_scale"] = qc, qsc
    ro, rl = oracle.attn_rows(host)
    B, Hq = len(lens), 64
    _gpu.assert_close(res["out"].float().cpu().numpy(), res["lse"].cpu().numpy(), ro.reshape(B, Hq, 128),
                      rl.reshape(B, Hq), case, "prologue -> attention")
