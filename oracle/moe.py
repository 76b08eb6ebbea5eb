"""Plain, slow CPU oracle of the clustered, compressed MoE layer forward pass.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the product path may import it.

Sources (page title, section):
  [T]  "Breaking the MoE LLM Trilemma: Dynamic Expert Clustering with Structured Compression"
       (paper notes): overall framework; key design 2 (shared base + low-rank residual, W~ eq.,
       factored forward, compression ratio CR); key design 3 (hierarchical routing: group first,
       then an expert inside the chosen group); key design 4 (FP16 base / INT4 residual).
  [R]  "混合专家模型的路由机制与工程落地" (routing mechanisms and engineering of MoE): section 1.2
       (FFN = W2 Act(W1 x) with Act = SwiGLU at Llama-3 dims; y = sum_i G_i(x) E_i(x));
       section 3.1 (router computed in FP32, experts in BF16/FP16); section 5.3 (dropless).
  [W]  "MoE架构演进白皮书" (MoE architecture whitepaper): chapter 1 top-2 code (top-k of the
       logits, then softmax over the selected logits); section 3.2 INT4 unpack convention.

Readings of points the pages leave open (each also listed in the design notes):
  * residual factor order: W~_i = W_base^g + B_i A_i^T, A_i in R^{d_in x r}, B_i in R^{d_out x r};
    the notes print A_i B_i^T and A_i (B_i^T x), which do not type-check against W x.
  * router arithmetic: FP32 per [R] 3.1, in the canonical order of ``canonical_logits`` so that
    routing indices are reproducible bit for bit.
  * level 2 is restricted to the chosen group(s) [T key design 3]; gate = p_g * q_e with p the
    softmax over the k_g selected group logits and q the softmax over the k_e selected expert
    logits inside that group [W ch. 1].  Ties: the lower index wins.
  * expert FFN = W~_down (silu(W~_gate x) * (W~_up x)) (SwiGLU, [R] 1.2), every matrix with its own
    residual; no capacity limit (dropless).
Floating point: everything after the router is FP64.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

LANES = 32      # canonical router: number of partial sums
CHUNK = 4       # canonical router: consecutive elements owned by one partial sum per block
BLOCK = LANES * CHUNK


# --------------------------------------------------------------------------------------------
# Router
# --------------------------------------------------------------------------------------------
def canonical_logits(x: np.ndarray, w: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """FP32 router logits s[t, j] = x_t . w_j (+ b_j) in the canonical order.

    [R] section 3.1 fixes only that the router runs in FP32; the order is this build's reading:
      partial sum l (l = 0..31) owns elements i with (i mod 128) div 4 == l and adds them in
      ascending i, each step s_l <- fl32(s_l + fl32(x_i * w_i));
      then for o = 16, 8, 4, 2, 1:  s_l <- fl32(s_l + s_{l xor o});
      logit = fl32(s_0 + b).
    x: [T, d] and w: [R, d] hold the exact input values (float32); d % 128 == 0.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, d = x.shape
    R = w.shape[0]
    assert d % BLOCK == 0, "canonical router order needs d % 128 == 0"
    nb = d // BLOCK
    xb = x.reshape(T, nb, LANES, CHUNK)
    wb = w.reshape(R, nb, LANES, CHUNK)
    s = np.zeros((T, R, LANES), dtype=np.float32)
    for j in range(nb):
        for u in range(CHUNK):
            prod = xb[:, None, j, :, u] * wb[None, :, j, :, u]   # fp32 products, rounded once
            s = s + prod                                          # fp32 add, rounded once
    lane = np.arange(LANES)
    for o in (16, 8, 4, 2, 1):
        s = s + s[:, :, lane ^ o]
    out = s[:, :, 0]
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float32)[None, :]
    return out.astype(np.float32)


def _softmax64(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    e = np.exp(v - v.max())
    return e / e.sum()


def _topk_desc(vals: np.ndarray, ids: np.ndarray, k: int) -> np.ndarray:
    """The k ids with the largest values; equal values -> lower id first. Ordered best first."""
    order = sorted(range(len(ids)), key=lambda i: (-float(vals[i]), int(ids[i])))
    return np.array([ids[i] for i in order[:k]], dtype=np.int64)


def route(x, w_group, b_group, w_expert, group_map, kg: int, ke: int, mode: str = "within") -> Dict[str, np.ndarray]:
    """Two-level routing [T key design 3] with top-k-then-softmax gates [W ch. 1].

    Level 1: group logits s_g (+ b_g); the kg best groups.  Level 2: inside each chosen group g,
    the ke best experts among {e : group_map[e] == g} by expert logit.
    Slots: group rank major, then expert rank; gate[t, slot] = p_g * q_e.
    Returns gidx [T,kg] int32, eidx [T,kg*ke] int32, gate [T,kg*ke] float64, and the FP32 logits.

    mode "across" is the other reading of the fine-grained workload's "top-3 experts across the
    chosen groups": the ke best experts over the union of the chosen groups' members (by expert
    logit, ties to the lower id), gates = softmax over those ke logits ([W ch. 1]: top-k, then
    softmax), the group gates p unused.  The slot layout stays the within-group one -- each chosen
    group's ke best members, which contain every member of the union's top ke -- and the slots
    that the union's top ke does not pick get gate 0 (so they add nothing to y).  ``active``
    [T, kg*ke] marks the picked slots.
    """
    group_map = np.asarray(group_map, dtype=np.int64)
    sg = canonical_logits(x, w_group, b_group)
    se = canonical_logits(x, w_expert, None)
    T = sg.shape[0]
    G = sg.shape[1]
    members = [np.nonzero(group_map == g)[0] for g in range(G)]
    gidx = np.zeros((T, kg), dtype=np.int32)
    eidx = np.zeros((T, kg * ke), dtype=np.int32)
    gate = np.zeros((T, kg * ke), dtype=np.float64)
    all_g = np.arange(G)
    for t in range(T):
        gs = _topk_desc(sg[t], all_g, kg)
        p = _softmax64(sg[t, gs])
        gidx[t] = gs
        for j, g in enumerate(gs):
            es = _topk_desc(se[t, members[g]], members[g], ke)
            q = _softmax64(se[t, es])
            eidx[t, j * ke:(j + 1) * ke] = es
            gate[t, j * ke:(j + 1) * ke] = p[j] * q
    active = np.ones((T, kg * ke), dtype=bool)
    if mode == "across":
        for t in range(T):
            union = np.concatenate([members[g] for g in gidx[t]])
            top = _topk_desc(se[t, union], union, ke)
            q = _softmax64(se[t, top])
            gate[t] = 0.0
            active[t] = False
            for i, e in enumerate(top):
                slot = int(np.nonzero(eidx[t] == e)[0][0])
                gate[t, slot] = q[i]
                active[t, slot] = True
    elif mode != "within":
        raise ValueError(mode)
    return {"gidx": gidx, "eidx": eidx, "gate": gate, "active": active, "group_logits": sg, "expert_logits": se}


# --------------------------------------------------------------------------------------------
# Dispatch order (the single-device form of the two-level dispatch of [T key design 3])
# --------------------------------------------------------------------------------------------
def permute(eidx: np.ndarray, group_map: np.ndarray, G: int, ke: int) -> Dict[str, np.ndarray]:
    """Stable orders of the routed work.

    Assignments a = t*k + slot sorted by key (group, expert, token):
      perm[i] = a, inv_pos[a] = i, expert_begin/expert_count [E], group_begin [G+1].
    (token, group-slot) rows sorted by key (group, token):
      row_asg[i] = t*kg + j, row_of[t*kg + j] = i, row_begin [G+1].
    """
    eidx = np.asarray(eidx, dtype=np.int64)
    group_map = np.asarray(group_map, dtype=np.int64)
    T, k = eidx.shape
    kg = k // ke
    E = group_map.shape[0]
    t_of = np.repeat(np.arange(T), k)
    e_of = eidx.reshape(-1)
    g_of = group_map[e_of]
    perm = np.array(sorted(range(T * k), key=lambda a: (g_of[a], e_of[a], t_of[a])), dtype=np.int64)
    inv_pos = np.empty(T * k, dtype=np.int64)
    inv_pos[perm] = np.arange(T * k)
    expert_count = np.bincount(e_of, minlength=E)
    # start of expert e = number of assignments whose (group, expert) key sorts before (g(e), e)
    expert_begin = np.array([np.count_nonzero((g_of < group_map[e]) | ((g_of == group_map[e]) & (e_of < e)))
                             for e in range(E)], dtype=np.int64)
    group_count = np.bincount(g_of, minlength=G)
    group_begin = np.concatenate([[0], np.cumsum(group_count)])

    row_t = np.repeat(np.arange(T), kg)
    row_j = np.tile(np.arange(kg), T)
    row_g = group_map[eidx[row_t, row_j * ke]] if T else np.zeros(0, dtype=np.int64)
    row_asg = np.array(sorted(range(T * kg), key=lambda a: (row_g[a], row_t[a])), dtype=np.int64)
    row_of = np.empty(T * kg, dtype=np.int64)
    row_of[row_asg] = np.arange(T * kg)
    row_begin = np.concatenate([[0], np.cumsum(np.bincount(row_g, minlength=G))])
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return {"perm": i32(perm), "inv_pos": i32(inv_pos), "expert_begin": i32(expert_begin),
            "expert_count": i32(expert_count), "group_begin": i32(group_begin),
            "row_asg": i32(row_asg), "row_of": i32(row_of), "row_begin": i32(row_begin)}


# --------------------------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------------------------
def dequant_int4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """INT4 group-64 rank rows -> FP64 [..., n].

    Byte j holds element 2j in its high nibble and 2j+1 in its low nibble; value = (u - 8) * s,
    s the FP16 scale of the element's 64-element group ([W] section 3.2 unpack convention:
    even offset -> high nibble, zero point 8; [T] key design 4: INT4 residual).
    """
    packed = np.asarray(packed, dtype=np.uint8)
    hi = (packed >> 4).astype(np.int64)
    lo = (packed & 0x0F).astype(np.int64)
    n = packed.shape[-1] * 2
    u = np.empty(packed.shape[:-1] + (n,), dtype=np.int64)
    u[..., 0::2] = hi
    u[..., 1::2] = lo
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    s = np.repeat(s, 64, axis=-1)
    return (u - 8).astype(np.float64) * s


def resid_dense(resid_m: dict, e: int) -> tuple:
    """(A^T [r, d_in], B^T [r, d_out]) of expert e in FP64 (dequantised when INT4)."""
    if "A" in resid_m:
        return (np.asarray(resid_m["A"][e], dtype=np.float64),
                np.asarray(resid_m["B"][e], dtype=np.float64))
    return (dequant_int4(resid_m["Aq"][e], resid_m["As"][e]),
            dequant_int4(resid_m["Bq"][e], resid_m["Bs"][e]))


def materialise(w_base_g: np.ndarray, At: np.ndarray, Bt: np.ndarray) -> np.ndarray:
    """W~ = W_base^g + B A^T explicitly, FP64 [d_out, d_in] ([T] key design 2, W~ equation)."""
    W = np.array(w_base_g, dtype=np.float64)
    if At.shape[0]:
        W += Bt.T @ At
    return W


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------------------------------------
# Forward
# --------------------------------------------------------------------------------------------
def _np(t):
    """torch CPU tensor or array -> numpy (BF16 widened exactly to FP32)."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch
        if t.dtype == torch.bfloat16 or t.dtype == torch.float16:
            t = t.float()
        return t.detach().cpu().numpy()
    return np.asarray(t)


def forward_tokens(inp: dict, tokens: Optional[Sequence[int]] = None, routing: Optional[dict] = None):
    """y_t = sum over the token's (g, e) of gate_{t,e} * W~_down,e (silu(W~_gate,e x_t) * W~_up,e x_t).

    ([R] 1.2 MoE sum with the SwiGLU FFN; [T] key design 2 expert parameterisation with every W~
    materialised explicitly.)  ``tokens`` selects a subset of rows (all when None); the routing is
    computed for every token either way.  Returns (y [n, d] FP64, routing dict).
    """
    cfg = inp["cfg"]
    x = _np(inp["x"]).astype(np.float32)
    if routing is None:
        routing = route(x, _np(inp["w_group"]), _np(inp["b_group"]), _np(inp["w_expert"]),
                         _np(inp["group_map"]), cfg.kg, cfg.ke, getattr(cfg, "route", "within"))
    toks = np.arange(cfg.T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    eidx = routing["eidx"][toks]
    gate = routing["gate"][toks]
    group_map = _np(inp["group_map"]).astype(np.int64)
    xs = x[toks].astype(np.float64)
    y = np.zeros((toks.size, cfg.d), dtype=np.float64)
    wg, wu, wd = (_np(inp["w_gate"]), _np(inp["w_up"]), _np(inp["w_down"]))
    resid = {m: {kk: _np(v) for kk, v in inp["resid"][m].items()} for m in ("gate", "up", "down")}
    for e in np.unique(eidx):
        rows, slots = np.nonzero(eidx == e)
        g = int(group_map[e])
        Wt = {}
        for m, base in (("gate", wg), ("up", wu), ("down", wd)):
            At, Bt = resid_dense(resid[m], int(e))
            Wt[m] = materialise(base[g], At, Bt)
        xe = xs[rows]
        h = silu(xe @ Wt["gate"].T) * (xe @ Wt["up"].T)
        out = h @ Wt["down"].T
        y[rows] += gate[rows, slots][:, None] * out
    return y, routing


def forward(inp: dict):
    """Whole-layer oracle: routing, dispatch orders and y for every token."""
    y, routing = forward_tokens(inp)
    cfg = inp["cfg"]
    perm = permute(routing["eidx"], _np(inp["group_map"]), cfg.G, cfg.ke)
    return {"y": y, **routing, **perm}


# --------------------------------------------------------------------------------------------
# Parameter accounting ([T] key design 2, compression ratio)
# --------------------------------------------------------------------------------------------
def compression_ratio(d_in: int, d_out: int, K: int, r: int) -> float:
    """CR = K d_in d_out / (d_in d_out + K r (d_in + d_out)): K dense experts vs one base + K rank-r residuals."""
    return K * d_in * d_out / (d_in * d_out + K * r * (d_in + d_out))


def param_counts(d: int, f: int, E: int, G: int, r: int) -> Dict[str, int]:
    """Stored parameters of a SwiGLU MoE layer: E dense experts vs G bases + E rank-r residuals."""
    per_dense = 3 * d * f
    per_resid = 3 * r * (d + f)
    return {"standard": E * per_dense, "clustered": G * per_dense + E * per_resid}
