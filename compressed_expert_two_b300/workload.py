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
