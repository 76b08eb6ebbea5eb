"""Plain CPU oracle of the compression step that produces the layer's weights.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product path imports it.

Source: "Breaking the MoE LLM Trilemma: Dynamic Expert Clustering with Structured Compression"
(paper notes), key design 2 (shared base + low-rank residual): the base of group g is the mean of
its experts' weights, each expert keeps a rank-r residual initialised by a truncated SVD of
(W_i - W_base^g), and the Frobenius reconstruction error is the quality measure; key design 4
(heterogeneous precision): the base stays 16-bit, the residual factors go to INT4.

Readings of points the notes leave open (each also listed in the design notes):
  * the mean is taken in FP32 in a fixed order -- s <- fl32(s + W_i) over the group's members in
    ascending expert id, then fl32(s / K) -- and stored as BF16 (round to nearest even), the base
    precision of the layer's workloads; the 16-bit code is decided in FP32 on both sides;
  * the residual is taken against the STORED (BF16) base, R_i = W_i - bf16(base), so that
    base + B A^T reconstructs W_i as well as the stored base allows;
  * the truncated SVD is the best rank-r approximation (Eckart-Young), R ~ U_r S_r V_r^T, split
    evenly between the factors: B = U_r S_r^{1/2} (d_out x r), A = V_r S_r^{1/2} (d_in x r), so that
    W~ = W_base + B A^T and both factors have the same scale before quantisation;
  * INT4 group-64 quantisation of the rank-major rows A^T [r][d_in] and B^T [r][d_out] in FP32:
    scale = fp16(absmax / 7) (round to nearest even), q = clamp(round_half_even(w / scale), -7, 7)
    (q = 0 when the scale is 0), nibble u = q + 8, element 2j in the high nibble of byte j (the
    layer's INT4 format, whitepaper section 3.2 unpack convention);
  * reconstruction error of expert i: ||W_i - W~_i||_F / ||W_i||_F with W~_i built from the
    stored base and the dequantised factors, in FP64.
Floating point: FP64 except where a stored code is decided (the base's BF16 value, the INT4
codes and FP16 scales), which follows the FP32 steps above exactly.
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np


def bf16_round(v: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 value (round to nearest, ties to even), returned as FP32."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def group_mean_base(W: np.ndarray, group_map: np.ndarray, G: int) -> np.ndarray:
    """W_base^g = (1/K) sum_{i in group g} W_i  (key design 2, base equation), in FP32 over the
    members in ascending id, stored as BF16 (returned as FP32 values).  W: [E][d_out][d_in]."""
    W = np.asarray(W, dtype=np.float32)
    group_map = np.asarray(group_map)
    out = np.empty((G,) + W.shape[1:], dtype=np.float32)
    for g in range(G):
        members = np.nonzero(group_map == g)[0]            # ascending ids
        s = np.zeros(W.shape[1:], dtype=np.float32)
        for e in members:
            s = (s + W[e]).astype(np.float32)             # one FP32 rounding per add
        out[g] = bf16_round((s / np.float32(len(members))).astype(np.float32))
    return out


def tsvd(R: np.ndarray, r: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Best rank-r approximation of R [d_out][d_in] (FP64 SVD): returns (B [d_out][r],
    A [d_in][r], sigma [r]) with B A^T = U_r S_r V_r^T and B = U_r S^{1/2}, A = V_r S^{1/2}."""
    U, S, Vt = np.linalg.svd(np.asarray(R, dtype=np.float64), full_matrices=False)
    root = np.sqrt(S[:r])
    return U[:, :r] * root[None, :], Vt[:r].T * root[None, :], S[:r]


def quantise_int4_g64(v: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Rank-major rows v [..., n] (n % 64 == 0, FP32 values) -> (codes uint8 [..., n/2],
    scales fp16 [..., n/64]) in the layer's INT4 group-64 format (FP32 decisions, see above)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    n = v.shape[-1]
    assert n % 64 == 0
    g = v.reshape(v.shape[:-1] + (n // 64, 64))
    amax = np.abs(g).max(axis=-1)
    scale = (amax / np.float32(7.0)).astype(np.float32).astype(np.float16)
    s32 = scale.astype(np.float32)[..., None]
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    q = np.where(s32 > 0, np.rint((g / safe).astype(np.float32)), np.float32(0.0))
    q = np.clip(q, -7, 7).astype(np.int64).reshape(v.shape)
    u = (q + 8).astype(np.uint8)
    codes = ((u[..., 0::2] << 4) | u[..., 1::2]).astype(np.uint8)
    return codes, scale


def reconstruction_error(W_i: np.ndarray, base_g: np.ndarray, At: np.ndarray, Bt: np.ndarray) -> float:
    """||W_i - (W_base + B A^T)||_F / ||W_i||_F in FP64 (At [r][d_in], Bt [r][d_out])."""
    W = np.asarray(W_i, dtype=np.float64)
    Wt = np.asarray(base_g, dtype=np.float64) + np.asarray(Bt, dtype=np.float64).T @ np.asarray(At, dtype=np.float64)
    return float(np.linalg.norm(W - Wt) / np.linalg.norm(W))


def compress_matrix(W: np.ndarray, group_map: np.ndarray, G: int, r: int) -> Dict[str, np.ndarray]:
    """The whole step for one matrix kind (gate, up or down) of every expert: W [E][d_out][d_in]
    -> base [G][d_out][d_in] (BF16 values), INT4 factors of A^T [E][r][d_in] and B^T [E][r][d_out],
    the singular values kept [E][r], and the reconstruction error of each expert."""
    from .moe import dequant_int4
    W = np.asarray(W, dtype=np.float32)
    E = W.shape[0]
    group_map = np.asarray(group_map)
    base = group_mean_base(W, group_map, G)
    out = {"base": base, "sigma": np.zeros((E, r)), "err": np.zeros(E)}
    Aq, As, Bq, Bs = [], [], [], []
    for e in range(E):
        R = W[e].astype(np.float64) - base[group_map[e]].astype(np.float64)
        B, A, S = tsvd(R, r)
        aq, a_s = quantise_int4_g64(A.T.astype(np.float32))
        bq, b_s = quantise_int4_g64(B.T.astype(np.float32))
        Aq.append(aq); As.append(a_s); Bq.append(bq); Bs.append(b_s)
        out["sigma"][e] = S
        out["err"][e] = reconstruction_error(W[e], base[group_map[e]], dequant_int4(aq, a_s), dequant_int4(bq, b_s))
    out.update(Aq=np.stack(Aq), As=np.stack(As), Bq=np.stack(Bq), Bs=np.stack(Bs))
    return out
