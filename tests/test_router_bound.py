"""The error bound the tensor-core router verifies its decisions with (CPU, no GPU).

The tensor-core router accepts a token's decision only when every pick's interval
[s - delta, s + delta] clears the next candidate's, with
    delta = c(d) * ||x|| * ||w|| + 2^-22 |s|,  c(d) = 1.01 ((d/8 + 8) 2^-22 + (d/32 + 6) 2^-24)
(the constant of the router kernel).  This checks the bound against the canonical FP32 order of
the oracle and against FP32 sums in other orders a tensor core may use: 16-product blocks summed
exactly and added into an FP32 accumulator rounded to nearest or truncated, in one accumulator or
in four interleaved ones; and the harsher alignment model, in which every product of a 16-deep
step and the accumulator are first aligned to the largest exponent among them and truncated to a
24-bit significand (no guard bits), then summed and truncated to FP32.  Every such sum must lie
within delta of the canonical logit, on Gaussian rows and on rows built to make the alignment
model lose the most (x = w, the first products large and all later ones just below the
accumulator's last bit, so that each is dropped).
"""
import math

import numpy as np
import pytest

import oracle


def c_err(d: int) -> float:
    return 1.01 * ((d / 8 + 8) * 2.0 ** -22 + (d / 32 + 6) * 2.0 ** -24)


def to_f32(v: np.ndarray, mode: str) -> np.ndarray:
    """FP64 -> FP32, round to nearest or toward zero."""
    f = v.astype(np.float32)
    if mode == "rz":
        over = np.abs(f.astype(np.float64)) > np.abs(v)
        f = np.where(over, np.nextafter(f, np.float32(0)), f)
    return f


def blocked_sum(x: np.ndarray, w: np.ndarray, mode: str, n_acc: int) -> np.ndarray:
    """sum_i x_i w_i: exact 16-product blocks, added into n_acc FP32 accumulators in turn
    (block b into accumulator b mod n_acc), each add rounded by `mode`; the accumulators are
    summed in FP32 at the end."""
    d = x.shape[1]
    prod = x.astype(np.float64)[:, None, :] * w.astype(np.float64)[None, :, :]   # exact
    blocks = prod.reshape(prod.shape[0], prod.shape[1], d // 16, 16).sum(-1)     # exact enough
    acc = np.zeros((n_acc,) + blocks.shape[:2], dtype=np.float32)
    for b in range(blocks.shape[2]):
        a = b % n_acc
        acc[a] = to_f32(acc[a].astype(np.float64) + blocks[:, :, b], mode)
    out = acc[0]
    for a in range(1, n_acc):
        out = (out + acc[a]).astype(np.float32)
    return out


def bf16(a: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (nearest even), kept as FP32."""
    u = a.astype(np.float32).view(np.uint32)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32)


@pytest.mark.parametrize("d", [256, 1024, 4096])
@pytest.mark.parametrize("mode,n_acc", [("rn", 1), ("rz", 1), ("rz", 4)])
def test_tensor_core_orders_stay_inside_the_bound(d, mode, n_acc):
    rng = np.random.default_rng(d + n_acc)
    x = bf16(rng.standard_normal((24, d)).astype(np.float32))
    w = bf16((rng.standard_normal((12, d)) / math.sqrt(d)).astype(np.float32))
    x[0] *= 1e3                                          # a large token
    w[1] = np.abs(w[1])                                  # a row with a large sum|x w| / |s| ratio
    canon = oracle.canonical_logits(x, w).astype(np.float64)
    other = blocked_sum(x, w, mode, n_acc).astype(np.float64)
    delta = c_err(d) * np.linalg.norm(x.astype(np.float64), axis=1)[:, None] * \
        np.linalg.norm(w.astype(np.float64), axis=1)[None, :] + 2.0 ** -22 * np.abs(other)
    diff = np.abs(other - canon)
    assert np.all(diff <= delta)
    # and the bound is not vacuous: the realised differences use a small part of it
    assert diff.max() <= 0.05 * delta.max()


def aligned_sum(x: np.ndarray, w: np.ndarray, n_acc: int, guard: int = 0) -> np.ndarray:
    """sum_i x_i w_i where each 16-deep step aligns its 16 exact products and the accumulator to
    the largest exponent among them, truncates each to 24 + guard significand bits, adds them
    exactly and truncates the result to FP32 (block b into accumulator b mod n_acc)."""
    d = x.shape[1]
    prod = x.astype(np.float64)[:, None, :] * w.astype(np.float64)[None, :, :]
    acc = np.zeros((n_acc,) + prod.shape[:2], dtype=np.float64)
    for b in range(d // 16):
        a = b % n_acc
        terms = np.concatenate([acc[a][..., None], prod[..., 16 * b:16 * b + 16]], axis=-1)
        _, e = np.frexp(np.abs(terms).max(-1))
        lsb = np.ldexp(1.0, e - 24 - guard)[..., None]
        acc[a] = to_f32((np.trunc(terms / lsb) * lsb).sum(-1), "rz").astype(np.float64)
    out = acc[0].astype(np.float32)
    for a in range(1, n_acc):
        out = (out + acc[a].astype(np.float32)).astype(np.float32)
    return out


def dropping_rows(d: int) -> np.ndarray:
    """Rows for which the alignment model drops every later product: x = w, the first 16 (one
    accumulator) or 64 (all four) elements 8, the rest sqrt(0.97 ulp(16 * 64))."""
    rows = []
    for n_big in (16, 64):
        r = np.full(d, math.sqrt(0.97 * 16 * 64 * 2.0 ** -23), dtype=np.float32)
        r[:n_big] = 8.0
        rows.append(bf16(r))
    return np.stack(rows)


@pytest.mark.parametrize("d", [256, 2048, 4096])
def test_alignment_truncation_model_stays_inside_the_bound(d):
    rng = np.random.default_rng(7 * d)
    gauss = bf16(rng.standard_normal((6, d)).astype(np.float32))
    drop = dropping_rows(d)
    for x, w in ((gauss, bf16((rng.standard_normal((5, d)) / math.sqrt(d)).astype(np.float32))), (drop, drop)):
        canon = oracle.canonical_logits(x, w).astype(np.float64)
        other = aligned_sum(x, w, 4).astype(np.float64)
        delta = c_err(d) * np.linalg.norm(x.astype(np.float64), axis=1)[:, None] * \
            np.linalg.norm(w.astype(np.float64), axis=1)[None, :] + 2.0 ** -22 * np.abs(other)
        assert np.all(np.abs(other - canon) <= delta)
    # the dropping rows do push the model near the bound (about 0.5 of delta at d = 256, 0.88 at 4096)
    canon = oracle.canonical_logits(drop, drop).astype(np.float64)
    other = aligned_sum(drop, drop, 4).astype(np.float64)
    n = np.linalg.norm(drop.astype(np.float64), axis=1)
    frac = np.abs(np.diag(other - canon)) / (c_err(d) * n * n + 2.0 ** -22 * np.abs(np.diag(other)))
    assert frac.max() >= 0.4
