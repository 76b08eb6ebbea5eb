"""Pins of the compression oracle (oracle/compress.py) to things other than itself (no GPU).

The step ("Breaking the MoE LLM Trilemma", paper notes, key design 2): group-mean base, truncated
SVD of each expert's residual, INT4 group-64 factors (key design 4), Frobenius reconstruction
error.  Each pin below would fail on a plausible mistake: a different summation order for the
mean, a transposed or unbalanced factor split, a wrong nibble order or rounding rule.
"""
import json
import os

import numpy as np
import torch

import oracle
from oracle import compress as C
from synth import CompressConfig, make_dense_experts, pack_int4_g64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_group_mean_exact_integers_and_membership():
    """Small integers: every FP32 sum is exact, so the base is the integer mean (here a multiple
    of 1/4, exact in BF16), taken over the right members (group map = seeded permutation)."""
    rng = np.random.default_rng(1)
    E, G = 8, 2
    W = rng.integers(-20, 20, size=(E, 4, 128)).astype(np.float32)
    gm = np.array([1, 0, 0, 1, 1, 0, 1, 0])
    base = C.group_mean_base(W, gm, G)
    for g in range(G):
        want = W[gm == g].astype(np.float64).mean(axis=0)
        assert np.array_equal(base[g].astype(np.float64), want)


def test_group_mean_order_and_rounding():
    """Members 0..3 hold 2^24, 1, 1, -2^24 at one element.  In ascending member order FP32 gives
    2^24 + 1 = 2^24 (tie to even), + 1 = 2^24, - 2^24 = 0: base 0 (the exact mean is 0.5, and the
    order 1, 1, 2^24, -2^24 would give 0.5).  A mean of 1/3 rounds to BF16 0.333984375."""
    W = np.zeros((4, 1, 128), dtype=np.float32)
    W[:, 0, 0] = [2.0 ** 24, 1.0, 1.0, -2.0 ** 24]
    W[:, 0, 1] = [1.0, 0.0, 0.0, 0.0]
    base = C.group_mean_base(W, np.zeros(4, dtype=np.int64), 1)
    assert base[0, 0, 0] == 0.0
    assert base[0, 0, 1] == 0.25
    W3 = np.zeros((3, 1, 128), dtype=np.float32)
    W3[0, 0, 0] = 1.0
    assert C.group_mean_base(W3, np.zeros(3, dtype=np.int64), 1)[0, 0, 0] == 0.333984375


def test_tsvd_on_a_constructed_spectrum():
    """R = U diag(s) V^T with orthonormal U, V from QR and known s: the rank-r truncation keeps the r
    largest s (sigma returned in descending order), B A^T = U_r diag(s_r) V_r^T, and the split is
    balanced: column k of B and of A both have norm sqrt(s_k)."""
    rng = np.random.default_rng(2)
    U, _ = np.linalg.qr(rng.standard_normal((96, 40)))
    V, _ = np.linalg.qr(rng.standard_normal((64, 40)))
    s = np.sort(rng.uniform(0.1, 5.0, 40))[::-1].copy()
    perm = rng.permutation(40)                              # the spectrum in scrambled column order
    R = (U[:, perm] * s[perm]) @ V[:, perm].T
    B, A, sig = C.tsvd(R, 8)
    assert np.allclose(sig, s[:8], rtol=1e-12)
    assert np.allclose(B @ A.T, (U[:, :8] * s[:8]) @ V[:, :8].T, atol=1e-10)
    assert np.allclose(np.linalg.norm(B, axis=0), np.sqrt(s[:8]), rtol=1e-10)
    assert np.allclose(np.linalg.norm(A, axis=0), np.sqrt(s[:8]), rtol=1e-10)
    # a diagonal matrix keeps its r largest entries
    D = np.diag([3.0, -7.0, 1.0, 5.0])
    B, A, sig = C.tsvd(D, 2)
    assert np.allclose(sig, [7.0, 5.0]) and np.allclose(B @ A.T, np.diag([0.0, -7.0, 0.0, 5.0]), atol=1e-12)


def test_quantiser_matches_the_independent_packer_and_the_golden_codes():
    """The oracle's INT4 quantiser agrees with the input generator's packer (a separate torch
    implementation of the same format) on random rows with zeros and exact ties, and re-quantising
    the hand-worked golden codes (every group holds a code of magnitude 7) returns them."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((6, 256)) * 0.02).astype(np.float32)
    v[1] = 0.0                                              # zero scale -> code 8
    v[2, :64] = np.arange(-32, 32) * 0.5 / 7 * 3            # values on half-code ties
    q, s = C.quantise_int4_g64(v)
    tq, ts = pack_int4_g64(torch.from_numpy(v))
    assert np.array_equal(q, tq.numpy()) and np.array_equal(s.view(np.uint16), ts.numpy().view(np.uint16))
    # the golden file's first case (byte 163 holds 1.0 and -2.5 at scale 0.5), placed at the start
    # of a 64-element group whose largest magnitude is 7 codes (3.5), so the scale is 0.5 again
    case = json.load(open(os.path.join(GOLDEN, "int4_convention.json")))["cases"][0]
    grp = np.zeros((1, 64), dtype=np.float32)
    grp[0, :2] = case["values"]
    grp[0, 2] = 7 * case["scale"]
    q2, s2 = C.quantise_int4_g64(grp)
    assert q2[0, 0] == case["bytes"][0] and q2[0, 1] == 0xF8 and np.all(q2[0, 2:] == 0x88)
    assert float(s2[0, 0]) == case["scale"]


def test_one_expert_per_group_reconstructs_exactly():
    """K = 1: the mean is the expert itself, the residual is zero (scale 0, every code 8) and the
    reconstruction error is 0."""
    rng = np.random.default_rng(4)
    W = bf16(rng.standard_normal((3, 128, 128)))
    out = C.compress_matrix(W, np.arange(3), 3, 4)
    assert np.array_equal(out["base"], W)
    assert np.all(out["Aq"] == 0x88) and np.all(out["err"] == 0.0)


def test_compression_of_synthetic_experts():
    """Experts that share a group part and differ by rank-r deviations plus 1% noise: the error
    is above the noise floor and below what dropping the residual altogether gives."""
    cfg = CompressConfig("pin", E=8, G=2, d=128, f=256, r=16, seed=5)
    inp = make_dense_experts(cfg, kinds=("gate",))
    W = inp["gate"]["W"].float().numpy()
    gm = inp["group_map"].numpy()
    out = C.compress_matrix(W, gm, cfg.G, cfg.r)
    no_resid = [np.linalg.norm(W[e] - out["base"][gm[e]]) / np.linalg.norm(W[e]) for e in range(cfg.E)]
    assert np.all(out["err"] > 0.005) and np.all(out["err"] < 0.6 * np.array(no_resid))
    assert np.all(np.diff(out["sigma"], axis=1) <= 0)
