"""Checks that pin the oracle's fused prologue (RMS QK-norm, then rotary
embedding; HPC-Ops/SGLang blog, "A fused attention prologue") to facts fixed
outside it: torch's float64 RMSNorm, the rotation's invariants and the
relative-position property that defines rotary embeddings."""
import numpy as np
import torch

import oracle
from load_balanced_paged_02_gb300 import workloads as wl


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run(case):
    return oracle.rope_norm(bits(case["qkv"]), case["positions"].cpu().numpy(), case["cos_sin"].cpu().numpy(),
                            case["q_weight"].cpu().numpy(), case["k_weight"].cpu().numpy(), case["eps"],
                            case["num_q_heads"], case["num_kv_heads"])


def check_norm_at_position_zero():
    """At position 0 the rotation is the identity: outputs are torch's rms_norm."""
    c = wl.make_prologue_case([0, 0, 0], 16, 2, seed=1)
    q, k, v = run(c)
    x = c["qkv"].to(torch.float64)
    qw = c["q_weight"].to(torch.float64)
    kw = c["k_weight"].to(torch.float64)
    ref_q = torch.nn.functional.rms_norm(x[:, :16], (128,), qw, eps=c["eps"])
    ref_k = torch.nn.functional.rms_norm(x[:, 16:18], (128,), kw, eps=c["eps"])
    assert np.allclose(q, ref_q.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(k, ref_k.numpy(), rtol=0, atol=1e-12)
    assert np.array_equal(v, x[:, 18:].numpy())


def check_rotation_keeps_pair_norms():
    """Each (i, i+64) pair is rotated: its norm equals the normalised input's."""
    c = wl.make_prologue_case([5, 77, 1000, 4095], 8, 1, seed=2, max_pos=4096)
    q, k, _ = run(c)
    x = c["qkv"].to(torch.float64)
    n_q = torch.nn.functional.rms_norm(x[:, :8], (128,), c["q_weight"].to(torch.float64), eps=c["eps"]).numpy()
    n_k = torch.nn.functional.rms_norm(x[:, 8:9], (128,), c["k_weight"].to(torch.float64), eps=c["eps"]).numpy()
    for out, ref in ((q, n_q), (k, n_k)):
        pair_out = out[..., :64] ** 2 + out[..., 64:] ** 2
        pair_ref = ref[..., :64] ** 2 + ref[..., 64:] ** 2
        assert np.allclose(pair_out, pair_ref, rtol=1e-6, atol=1e-9)
        assert not np.allclose(out, ref, atol=1e-3), "positions > 0 must rotate"


def check_relative_position():
    """q(m) . k(n) depends only on m - n for the same q and k inputs."""
    rng = np.random.default_rng(3)
    for _ in range(8):
        m, n = (int(v) for v in rng.integers(0, 2000, size=2))
        d = int(rng.integers(0, 2000))
        base = wl.make_prologue_case([m, n], 8, 1, seed=4, max_pos=4096)
        shifted = dict(base, positions=torch.tensor([m + d, n + d], dtype=torch.int32))
        q0, k0, _ = run(base)
        q1, k1, _ = run(shifted)
        # token 0's query heads against token 1's key head
        s0 = q0[0] @ k0[1, 0]
        s1 = q1[0] @ k1[1, 0]
        assert np.allclose(s0, s1, rtol=0, atol=2e-4 * max(1.0, np.abs(s0).max())), (m, n, d)
