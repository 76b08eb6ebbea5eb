"""Algorithmic work of one layer forward pass (the roofline numerators).

FLOPs count the base product once per (token, group) row -- the reuse the layer is built for
("Breaking the MoE LLM Trilemma", key design 2: the base term is computed once for the group's
experts on the same tokens) -- the rank-r residual once per (token, expert), and the router once
for all G + E rows:
    F/token = 6 d f k_g + 6 r (d + f) k_g k_e + 2 d (G + E).
Bytes count every weight the pass needs exactly once, x read once and y written once:
    B = sum_{groups hit} 3 d f s_base + sum_{experts hit} 3 r (d + f) (1/2 + 2/64) + (G+E) d s_act
        + 2 T d s_act     (INT4 residual: half a byte per element + an FP16 scale per 64).
"""
from __future__ import annotations


def flops(cfg, T=None) -> float:
    T = cfg.T if T is None else T
    per_tok = 6 * cfg.d * cfg.f * cfg.kg + 6 * cfg.r * (cfg.d + cfg.f) * cfg.kg * cfg.ke \
        + 2 * cfg.d * (cfg.G + cfg.E)
    return float(per_tok) * T


def ffn_flops(cfg, T=None):
    """(gate/up GEMM flops, down GEMM flops) of the base+residual products."""
    T = cfg.T if T is None else T
    rows = T * cfg.kg
    up = 4.0 * cfg.d * cfg.f * rows + 4.0 * cfg.r * (cfg.d + cfg.f) * rows * cfg.ke
    down = 2.0 * cfg.d * cfg.f * rows + 2.0 * cfg.r * (cfg.d + cfg.f) * rows * cfg.ke
    return up, down


def bytes_moved(cfg, groups_hit: int, experts_hit: int, T=None) -> float:
    T = cfg.T if T is None else T
    s_act = 2 if cfg.dtype == "bf16" else 4
    s_res = (0.5 + 2.0 / 64) if cfg.resid == "int4" else 4.0
    return (groups_hit * 3.0 * cfg.d * cfg.f * s_act + experts_hit * 3.0 * cfg.r * (cfg.d + cfg.f) * s_res
            + (cfg.G + cfg.E) * cfg.d * s_act + 2.0 * T * cfg.d * s_act)


def kernel_work(cfg, kernel: str, groups_hit: int, experts_hit: int, T=None):
    """(algorithmic FLOPs, algorithmic DRAM bytes) of one launch of a named kernel.

    Rows R = T k_g.  Weights are counted once per launch at their stored size (BF16 base,
    INT4 + FP16-scale residual), activations once in and once out.
      ffn_up:   4 d f R (gate/up base) + 6 r f R k_e (B_gate U, B_up U, A_down^T h);
                bytes: gate/up bases of the groups hit, B_gate/B_up/A_down of the experts hit,
                X rows in, hsum rows out.
      ffn_down: 2 d f R (down base) + 2 r d R k_e (B_down v); bytes: down bases, B_down, hsum in, y out.
      u_gemm:   4 r d R k_e (A_gate^T x, A_up^T x); bytes: A_gate/A_up of the experts hit, X rows.
      router:   2 d (G + E) T; bytes: x and the router rows.
    Other kernels fall back to the whole-layer figures.
    """
    T = cfg.T if T is None else T
    R = T * cfg.kg
    s_act = 2 if cfg.dtype == "bf16" else 4
    s_res = (0.5 + 2.0 / 64) if cfg.resid == "int4" else 4.0
    d, f, r, ke = cfg.d, cfg.f, cfg.r, cfg.ke
    if kernel.startswith("ffn_up"):
        return (4.0 * d * f * R + 6.0 * r * f * R * ke,
                groups_hit * 2.0 * d * f * s_act + experts_hit * 3.0 * r * f * s_res + R * (d + f) * s_act)
    if kernel.startswith("ffn_down"):
        return (2.0 * d * f * R + 2.0 * r * d * R * ke,
                groups_hit * 1.0 * d * f * s_act + experts_hit * r * d * s_res + R * (d + f) * s_act)
    if kernel.startswith("u_gemm"):
        return 4.0 * r * d * R * ke, experts_hit * 2.0 * r * d * s_res + R * d * s_act
    if kernel.startswith("router"):
        return 2.0 * d * (cfg.G + cfg.E) * T, (T + cfg.G + cfg.E) * d * s_act
    return flops(cfg, T), bytes_moved(cfg, groups_hit, experts_hit, T)


def load_stats(gidx, eidx, G: int, E: int, active=None) -> dict:
    """Load balance of one batch's routing (the imbalance the clustering is meant to bound; the
    pages report load variance and the max/mean ratio): rows per group (one per token and chosen
    group) and assignments per expert, from the router's gidx [T][k_g] and eidx [T][k] (integer
    arrays or tensors); with ``active`` [T][k] (the across-groups reading's picked slots) only
    those assignments count.  max/mean is 1 for a perfectly even batch; cv = std/mean."""
    import numpy as np
    g = np.bincount(np.asarray(gidx).reshape(-1), minlength=G).astype(np.float64)
    ev = np.asarray(eidx).reshape(-1)
    if active is not None:
        ev = ev[np.asarray(active).reshape(-1).astype(bool)]
    e = np.bincount(ev, minlength=E).astype(np.float64)

    def summary(c):
        m = c.mean()
        return {"max_over_mean": float(c.max() / m) if m > 0 else 0.0,
                "cv": float(c.std() / m) if m > 0 else 0.0,
                "min": int(c.min()), "max": int(c.max())}

    return {"group": summary(g), "expert": summary(e)}
