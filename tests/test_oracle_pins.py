"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a value the pages print, a closed form, an invariant, a
textbook/library special case, or brute force on tiny inputs.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, MoEConfig, make_inputs, pack_int4_g64, variant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_cfg(**kw):
    base = dict(name="pin", T=8, d=128, f=64, E=8, G=2, kg=1, ke=2, r=4, dtype="f32", resid="f32",
                group_map="contiguous", seed=11)
    base.update(kw)
    return MoEConfig(**base)


# ------------------------------------------------------------------ canonical FP32 router order
def test_canonical_logits_exact_integer_sums():
    """Small integers: every partial sum is exact, so the result must equal the integer dot."""
    rng = np.random.default_rng(0)
    x = rng.integers(-3, 4, size=(5, 256)).astype(np.float32)
    w = rng.integers(-3, 4, size=(7, 256)).astype(np.float32)
    b = rng.integers(-5, 6, size=7).astype(np.float32)
    got = oracle.canonical_logits(x, w, b)
    want = x.astype(np.int64) @ w.astype(np.int64).T + b.astype(np.int64)
    assert np.array_equal(got.astype(np.int64), want)


def _one_hot_case(entries, d=256):
    x = np.zeros((1, d), dtype=np.float32)
    for i, v in entries.items():
        x[0, i] = v
    return x, np.ones((1, d), dtype=np.float32)


def test_canonical_logits_butterfly_order():
    """Hand-derived rounding: partial sums 0..3 hold 2^24, 1, 1, -2^24 (elements 0, 4, 8, 12).

    xor 16/8/4 add zeros; xor 2: s0 = fl(2^24 + 1) = 2^24 (tie to even), s1 = 1 - 2^24 (exact);
    xor 1: s0 = 2^24 + (1 - 2^24) = 1.  A left-to-right sum gives 0 and the exact sum is 2.
    """
    x, w = _one_hot_case({0: 2.0 ** 24, 4: 1.0, 8: 1.0, 12: -2.0 ** 24})
    assert oracle.canonical_logits(x, w)[0, 0] == 1.0


def test_canonical_logits_in_lane_order():
    """Elements 0, 1 (block 0) and 128, 129 (block 1) all belong to partial sum 0, added in
    ascending order: 2^24, +1 -> 2^24, +1 -> 2^24, -2^24 -> 0 (descending order would give 2)."""
    x, w = _one_hot_case({0: 2.0 ** 24, 1: 1.0, 128: 1.0, 129: -2.0 ** 24})
    assert oracle.canonical_logits(x, w)[0, 0] == 0.0
    # element 4 is in partial sum 1, so the same values spread over two sums give 2^24+1-2^24+1
    x, w = _one_hot_case({0: 2.0 ** 24, 4: 1.0, 128: 1.0, 132: -2.0 ** 24})
    # s0 = 2^24 + 1 -> 2^24 ; s1 = 1 - 2^24 ; s0 + s1 = 1
    assert oracle.canonical_logits(x, w)[0, 0] == 1.0


def test_canonical_logits_fp64_error_bound():
    rng = np.random.default_rng(1)
    d = 1024
    x = rng.standard_normal((64, d)).astype(np.float32)
    w = (rng.standard_normal((16, d)) / math.sqrt(d)).astype(np.float32)
    got = oracle.canonical_logits(x, w).astype(np.float64)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    mag = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
    n = d // 32 + 5 + 1
    assert np.all(np.abs(got - exact) <= n * 2.0 ** -24 * mag * 1.01)


def test_canonical_routing_differs_from_fp64_only_at_near_ties():
    """The canonical FP32 logits decide like exact (FP64) logits except where two candidates lie
    within the canonical order's rounding bound of each other: every token whose FP64 routing
    differs has such a near tie, and forcing exact ties (duplicated router rows) makes the lower
    index win in both."""
    rng = np.random.default_rng(3)
    T, d, G, K, kg, ke = 400, 256, 4, 4, 2, 2
    E = G * K
    gm = np.arange(E) // K
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((G, d)) / math.sqrt(d)).astype(np.float32)
    we = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
    we[5] = we[6]                                             # exact ties inside group 1
    r = oracle.route(x, wg, None, we, gm, kg, ke)
    ex_g = x.astype(np.float64) @ wg.astype(np.float64).T
    ex_e = x.astype(np.float64) @ we.astype(np.float64).T
    bound_g = (d // 32 + 6) * 2.0 ** -24 * (np.abs(x) @ np.abs(wg).T)
    bound_e = (d // 32 + 6) * 2.0 ** -24 * (np.abs(x) @ np.abs(we).T)
    def has_near_tie(vals, bnd, cands):
        return any(abs(vals[a] - vals[b]) <= bnd[a] + bnd[b] for a in cands for b in cands if a < b)

    for t in range(T):
        gs = sorted(range(G), key=lambda g: (-ex_g[t, g], g))[:kg]
        if gs != list(r["gidx"][t]):
            assert has_near_tie(ex_g[t], bound_g[t], range(G)), t
            continue
        for j, g in enumerate(gs):
            mem = list(np.nonzero(gm == g)[0])
            es = sorted(mem, key=lambda e: (-ex_e[t, e], e))[:ke]
            if es != list(r["eidx"][t, j * ke:(j + 1) * ke]):
                assert has_near_tie(ex_e[t], bound_e[t], mem), t
    # the duplicated rows: wherever both are picked, the lower id comes first
    for t in range(T):
        for j in range(kg):
            picks = list(r["eidx"][t, j * ke:(j + 1) * ke])
            if 5 in picks and 6 in picks:
                assert picks.index(5) < picks.index(6)


# ------------------------------------------------------------------ INT4 format
def test_int4_golden_convention():
    spec = json.load(open(os.path.join(GOLDEN, "int4_convention.json")))
    for case in spec["cases"]:
        b = np.full(32, 0x88, dtype=np.uint8)          # pad the 64-element group with zeros
        b[:len(case["bytes"])] = case["bytes"]
        s = np.array([case["scale"]], dtype=np.float16)
        v = oracle.dequant_int4(b, s)
        n = len(case["values"])
        assert np.array_equal(v[:n], np.array(case["values"]))
        assert np.all(v[n:] == 0)


def test_int4_pack_roundtrip_error_bound():
    g = torch.Generator().manual_seed(5)
    w = torch.randn(3, 5, 256, generator=g) * 0.02
    q, s = pack_int4_g64(w)
    back = oracle.dequant_int4(q.numpy(), s.numpy())
    step = np.repeat(s.float().numpy().astype(np.float64), 64, axis=-1)
    err = np.abs(back - w.double().numpy())
    # symmetric rounding to the nearest code: error <= step/2 (+ fp16 rounding of the scale)
    assert np.all(err <= 0.5 * step + 7 * step * 2.0 ** -10 + 1e-12)
    # and the nibble order matters: swapping the nibbles breaks the bound
    swapped = ((q.numpy() & 0x0F) << 4) | (q.numpy() >> 4)
    err2 = np.abs(oracle.dequant_int4(swapped, s.numpy()) - w.double().numpy())
    assert err2.max() > 2 * step.max()


# ------------------------------------------------------------------ routing
def test_gates_sum_to_one_and_group_gate_one():
    for name in ("tiny_f32",):
        inp = make_inputs(CONFIGS[name])
        cfg = inp["cfg"]
        r = oracle.route(oracle.moe._np(inp["x"]), oracle.moe._np(inp["w_group"]), None,
                         oracle.moe._np(inp["w_expert"]), inp["group_map"].numpy(), cfg.kg, cfg.ke)
        assert np.allclose(r["gate"].sum(1), 1.0, atol=1e-12, rtol=0)
    cfg = tiny_cfg(T=64, G=4, E=16, kg=2, ke=3)
    inp = make_inputs(cfg)
    r = oracle.route(oracle.moe._np(inp["x"]), oracle.moe._np(inp["w_group"]), None,
                     oracle.moe._np(inp["w_expert"]), inp["group_map"].numpy(), cfg.kg, cfg.ke)
    assert np.allclose(r["gate"].sum(1), 1.0, atol=1e-12, rtol=0)
    # experts of a slot group belong to that group and are distinct
    gm = inp["group_map"].numpy()
    for t in range(cfg.T):
        for j in range(cfg.kg):
            es = r["eidx"][t, j * cfg.ke:(j + 1) * cfg.ke]
            assert np.all(gm[es] == r["gidx"][t, j]) and len(set(es)) == cfg.ke


def test_two_groups_two_experts_hand_computed_gates():
    """k_g = 2, k_e = 2 on one token whose logits are small integers (x is one-hot, so every
    canonical logit is a router row's first entry, exactly).  Groups (G = 3, K = 3, contiguous):
    logits 2, 0, 1 -> groups 0 then 2, p = (e/(e+1), 1/(e+1)).  Group 0's experts 0, 1, 2 have
    logits 0, 3, 1 -> experts 1 then 2, q = (e^2/(e^2+1), 1/(e^2+1)).  Group 2's experts 6, 7, 8
    have logits -1, -1, 2 -> expert 8, then the tie between 6 and 7 goes to 6,
    q = (e^3/(e^3+1), 1/(e^3+1)).  gate = p_g q_e in slot order (group rank, then expert rank)."""
    d = 128
    x = np.zeros((1, d), dtype=np.float32)
    x[0, 0] = 1.0
    wg = np.zeros((3, d), dtype=np.float32)
    wg[:, 0] = [2, 0, 1]
    we = np.zeros((9, d), dtype=np.float32)
    we[:, 0] = [0, 3, 1, 5, 5, 5, -1, -1, 2]
    gm = np.repeat(np.arange(3), 3)
    r = oracle.route(x, wg, None, we, gm, 2, 2)
    e = math.e
    p0, p1 = e / (e + 1), 1 / (e + 1)
    assert r["gidx"].tolist() == [[0, 2]]
    assert r["eidx"].tolist() == [[1, 2, 8, 6]]
    want = [p0 * e ** 2 / (e ** 2 + 1), p0 / (e ** 2 + 1), p1 * e ** 3 / (e ** 3 + 1), p1 / (e ** 3 + 1)]
    assert np.allclose(r["gate"][0], want, rtol=0, atol=1e-15)
    assert abs(r["gate"][0].sum() - 1.0) < 1e-15


def test_across_groups_hand_computed_gates():
    """The token of the test above in the across-groups reading: groups 0 and 2 are chosen; the
    union of their members {0, 1, 2, 6, 7, 8} has logits 0, 3, 1, -1, -1, 2.  Top-2: experts 1 and
    8, gates softmax(3, 2) = (e/(e+1), 1/(e+1)); the within-group slots [1, 2, 8, 6] stay, with
    expert 2's and 6's gates 0.  Top-3: experts 1, 8, 2 with softmax(3, 2, 1); the slots are each
    group's top 3, [1, 2, 0, 8, 6, 7] (6 before 7: equal logits, lower id first)."""
    d = 128
    x = np.zeros((1, d), dtype=np.float32)
    x[0, 0] = 1.0
    wg = np.zeros((3, d), dtype=np.float32)
    wg[:, 0] = [2, 0, 1]
    we = np.zeros((9, d), dtype=np.float32)
    we[:, 0] = [0, 3, 1, 5, 5, 5, -1, -1, 2]
    gm = np.repeat(np.arange(3), 3)
    e = math.e
    r = oracle.route(x, wg, None, we, gm, 2, 2, "across")
    assert r["gidx"].tolist() == [[0, 2]] and r["eidx"].tolist() == [[1, 2, 8, 6]]
    assert np.allclose(r["gate"][0], [e / (e + 1), 0, 1 / (e + 1), 0], rtol=0, atol=1e-15)
    assert r["active"].tolist() == [[True, False, True, False]]
    r = oracle.route(x, wg, None, we, gm, 2, 3, "across")
    assert r["eidx"].tolist() == [[1, 2, 0, 8, 6, 7]]
    z = e * e + e + 1
    assert np.allclose(r["gate"][0], [e * e / z, 1 / z, 0, e / z, 0, 0], rtol=0, atol=1e-15)


def test_across_groups_brute_force_and_special_cases():
    """Brute force over every ke-subset of the union of the chosen groups' members (T = 8):
    the picked experts are the unique subset whose members all beat every other member of the
    union in (logit desc, id asc) order, and their gates are the softmax of their logits.  With
    k_g = 1 the union is one group and the reading equals the within-group one; with k_g = G it is
    a plain top-k over all experts (torch.topk / softmax)."""
    cfg = tiny_cfg(T=8, E=12, G=3, kg=2, ke=2)
    inp = make_inputs(cfg)
    x, wg, we = (oracle.moe._np(inp[k]) for k in ("x", "w_group", "w_expert"))
    gm = inp["group_map"].numpy()
    r = oracle.route(x, wg, None, we, gm, 2, 2, "across")
    se = r["expert_logits"]
    for t in range(cfg.T):
        union = [int(e) for g in r["gidx"][t] for e in np.nonzero(gm == g)[0]]
        before = lambda a, b: se[t, a] > se[t, b] or (se[t, a] == se[t, b] and a < b)
        winners = [set(S) for S in itertools.combinations(union, 2)
                   if all(before(a, b) for a in S for b in union if b not in S)]
        assert len(winners) == 1
        picked = {int(e) for e, on in zip(r["eidx"][t], r["active"][t]) if on}
        assert picked == winners[0]
        lg = np.array([se[t, e] for e in sorted(picked)], dtype=np.float64)
        want = dict(zip(sorted(picked), np.exp(lg - lg.max()) / np.exp(lg - lg.max()).sum()))
        for e, g, on in zip(r["eidx"][t], r["gate"][t], r["active"][t]):
            assert (g == 0.0) != on and (not on or abs(g - want[int(e)]) < 1e-15)
    within = oracle.route(x, wg, None, we, gm, 1, 3)
    across = oracle.route(x, wg, None, we, gm, 1, 3, "across")
    assert np.array_equal(within["eidx"], across["eidx"]) and np.allclose(within["gate"], across["gate"], atol=1e-15)
    r = oracle.route(x, wg, None, we, gm, 3, 2, "across")
    vals, idx = torch.topk(torch.from_numpy(se).double(), 2, dim=-1)
    for t in range(cfg.T):
        picked = [int(e) for e, on in zip(r["eidx"][t], r["active"][t]) if on]
        assert sorted(picked) == sorted(idx[t].tolist())
        gates = {int(e): g for e, g in zip(r["eidx"][t], r["gate"][t]) if g > 0}
        sm = torch.softmax(vals[t], -1).numpy()
        assert all(abs(gates[int(e)] - p) < 1e-15 for e, p in zip(idx[t].tolist(), sm))


def test_across_groups_output_brute_force():
    """y of the across reading equals the gated sum over the picked experts only, each computed
    independently in factored form."""
    cfg = tiny_cfg(T=6, E=12, G=3, kg=2, ke=2, route="across", resid_std=0.2)
    inp = make_inputs(cfg)
    y, r = oracle.forward_tokens(inp)
    for t in range(cfg.T):
        xt = inp["x"][t].double().numpy()
        want = sum(g * _expert_ffn_factored(inp, int(e), xt)
                   for e, g, on in zip(r["eidx"][t], r["gate"][t], r["active"][t]) if on)
        assert np.allclose(y[t], want, rtol=1e-10, atol=1e-12)


def test_route_matches_torch_topk_when_one_group():
    """G = 1: level 1 is trivial and level 2 is a plain top-k over all experts, softmax over the
    selected logits (library topk/softmax)."""
    cfg = tiny_cfg(T=32, E=8, G=1, kg=1, ke=3)
    inp = make_inputs(cfg)
    x = oracle.moe._np(inp["x"])
    r = oracle.route(x, oracle.moe._np(inp["w_group"]), None, oracle.moe._np(inp["w_expert"]),
                     inp["group_map"].numpy(), 1, 3)
    logits = torch.from_numpy(r["expert_logits"]).double()
    vals, idx = torch.topk(logits, 3, dim=-1)
    assert np.array_equal(r["eidx"], idx.numpy())
    assert np.allclose(r["gate"], torch.softmax(vals, -1).numpy(), rtol=0, atol=1e-15)


def _expert_ffn_factored(inp, e, xt):
    """Independent per-expert FFN in factored form W_base x + B (A^T x) (no materialisation)."""
    g = int(inp["group_map"][e])
    out = {}
    for m, base in (("gate", inp["w_gate"]), ("up", inp["w_up"])):
        At, Bt = oracle.resid_dense({k: v.numpy() for k, v in inp["resid"][m].items()}, e)
        out[m] = base[g].double().numpy() @ xt + Bt.T @ (At @ xt)
    h = out["gate"] / (1 + np.exp(-out["gate"])) * out["up"]
    At, Bt = oracle.resid_dense({k: v.numpy() for k, v in inp["resid"]["down"].items()}, e)
    return inp["w_down"][g].double().numpy() @ h + Bt.T @ (At @ h)


def test_brute_force_routing_and_output():
    """T=8, G=2, K=4, top-1 group then top-2: enumerate all 2 x 6 choices per token.  The chosen
    one is the unique choice whose picks beat every unpicked option, and y equals that choice's
    gated output (all other choices give different outputs)."""
    cfg = tiny_cfg()
    inp = make_inputs(cfg)
    y, r = oracle.forward_tokens(inp)
    gm = inp["group_map"].numpy()
    sg, se = r["group_logits"], r["expert_logits"]
    for t in range(cfg.T):
        xt = inp["x"][t].double().numpy()
        winners = []
        outs = []
        for g in range(cfg.G):
            mem = [e for e in range(cfg.E) if gm[e] == g]
            for pair in itertools.combinations(mem, 2):
                other_g = [h for h in range(cfg.G) if h != g]
                beats_g = all((sg[t, g], -g) > (sg[t, h], -h) for h in other_g)
                beats_e = all((se[t, e], -e) > (se[t, o], -o) for e in pair for o in mem if o not in pair)
                lv = np.array([se[t, e] for e in pair], dtype=np.float64)
                q = np.exp(lv - lv.max()); q /= q.sum()
                out = sum(q[i] * _expert_ffn_factored(inp, pair[i], xt) for i in range(2))
                outs.append(out)
                if beats_g and beats_e:
                    winners.append((g, set(pair), out))
        assert len(winners) == 1
        g, pair, out = winners[0]
        assert r["gidx"][t, 0] == g and set(r["eidx"][t]) == pair
        scale = np.abs(out).max()
        assert np.allclose(y[t], out, rtol=0, atol=1e-12 * scale)
        assert sum(np.allclose(y[t], o, rtol=0, atol=1e-9 * scale) for o in outs) == 1


# ------------------------------------------------------------------ permutation
def test_permute_invariants_and_lexsort():
    cfg = tiny_cfg(T=200, G=4, E=16, kg=2, ke=2, d=128, f=64, r=0)
    inp = make_inputs(cfg)
    r = oracle.route(oracle.moe._np(inp["x"]), oracle.moe._np(inp["w_group"]), None,
                     oracle.moe._np(inp["w_expert"]), inp["group_map"].numpy(), cfg.kg, cfg.ke)
    p = oracle.permute(r["eidx"], inp["group_map"].numpy(), cfg.G, cfg.ke)
    k = cfg.k
    gm = inp["group_map"].numpy()
    flat_e = r["eidx"].reshape(-1)
    perm = p["perm"]
    # bijection and inverse
    assert sorted(perm.tolist()) == list(range(cfg.T * k))
    assert np.array_equal(p["inv_pos"][perm], np.arange(cfg.T * k))
    keys = [(gm[flat_e[a]], flat_e[a], a // k) for a in perm]
    assert all(keys[i] < keys[i + 1] for i in range(len(keys) - 1))       # strictly increasing
    # library sort of the same keys
    ls = np.lexsort((np.repeat(np.arange(cfg.T), k), flat_e, gm[flat_e]))
    assert np.array_equal(ls, perm)
    # offsets
    assert p["expert_count"].sum() == cfg.T * k
    for e in range(cfg.E):
        seg = perm[p["expert_begin"][e]:p["expert_begin"][e] + p["expert_count"][e]]
        assert np.all(flat_e[seg] == e)
    assert p["group_begin"][-1] == cfg.T * k
    # rows (token, group slot) sorted by (group, token)
    rows = p["row_asg"]
    rg = gm[r["eidx"][rows // cfg.kg, (rows % cfg.kg) * cfg.ke]]
    rkeys = list(zip(rg, rows // cfg.kg))
    assert all(rkeys[i] < rkeys[i + 1] for i in range(len(rkeys) - 1))
    assert np.array_equal(p["row_of"][rows], np.arange(cfg.T * cfg.kg))
    assert np.array_equal(np.diff(p["row_begin"]), np.bincount(rg, minlength=cfg.G))


# ------------------------------------------------------------------ FFN special cases
def test_factor_identity():
    """W~ x == W_base x + B (A^T x) for every matrix of an INT4 expert."""
    cfg = tiny_cfg(dtype="bf16", resid="int4", d=256, f=128, r=16, resid_std=0.2)
    inp = make_inputs(cfg)
    rng = np.random.default_rng(3)
    xt = rng.standard_normal(256)
    for e in (0, 5):
        g = int(inp["group_map"][e])
        At, Bt = oracle.resid_dense({k: v.numpy() for k, v in inp["resid"]["gate"].items()}, e)
        W = oracle.materialise(inp["w_gate"][g].float().numpy(), At, Bt)
        lhs = W @ xt
        rhs = inp["w_gate"][g].double().numpy() @ xt + Bt.T @ (At @ xt)
        assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12 * np.abs(rhs).max())


def test_rank0_is_dense_group_base_moe():
    """r = 0 and one group per token: y_t = FFN_base^{g(t)}(x_t) whatever the expert choice (gates
    of the chosen group sum to 1).  Checked against torch FP64 silu/matmul."""
    cfg = tiny_cfg(T=32, r=0, dtype="bf16", resid="int4", d=256, f=128)
    inp = make_inputs(cfg)
    y, r = oracle.forward_tokens(inp)
    x = inp["x"].double()
    for t in range(cfg.T):
        g = int(r["gidx"][t, 0])
        a = torch.nn.functional.silu(inp["w_gate"][g].double() @ x[t]) * (inp["w_up"][g].double() @ x[t])
        want = inp["w_down"][g].double() @ a
        assert torch.allclose(torch.from_numpy(y[t]), want, rtol=1e-11, atol=1e-12)


def test_one_expert_per_group_rank0_is_textbook_topk_moe():
    """K = 1 (G = E), r = 0: the layer is a standard top-k MoE with router w_group and experts the
    bases, y = sum_i softmax(topk logits)_i FFN_i(x) (per-expert torch loop)."""
    cfg = tiny_cfg(T=24, E=6, G=6, kg=2, ke=1, r=0)
    inp = make_inputs(cfg)
    y, r = oracle.forward_tokens(inp)
    logits = torch.from_numpy(r["group_logits"]).double()
    vals, idx = torch.topk(logits, 2, dim=-1)
    gates = torch.softmax(vals, -1)
    x = inp["x"].double()
    for t in range(cfg.T):
        acc = torch.zeros(cfg.d, dtype=torch.float64)
        for j in range(2):
            e = int(idx[t, j])
            a = torch.nn.functional.silu(inp["w_gate"][e].double() @ x[t]) * (inp["w_up"][e].double() @ x[t])
            acc += gates[t, j] * (inp["w_down"][e].double() @ a)
        assert torch.allclose(torch.from_numpy(y[t]), acc, rtol=1e-11, atol=1e-12)


def test_residual_is_visible_in_amplified_variant():
    cfg = tiny_cfg(T=16, dtype="bf16", resid="int4", d=256, f=128, r=16)
    y_amp, _ = oracle.forward_tokens(make_inputs(variant(cfg, "amplified")))
    y_r0, _ = oracle.forward_tokens(make_inputs(variant(cfg.replace(resid_std=0.2), "rank0")))
    diff = np.abs(y_amp - y_r0).sum() / np.abs(y_r0).sum()
    assert diff > 0.05


# ------------------------------------------------------------------ parameter accounting
def test_compression_ratio_closed_form():
    spec = json.load(open(os.path.join(GOLDEN, "compression_ratio.json")))
    cr = oracle.compression_ratio(spec["d_in"], spec["d_out"], spec["K"], spec["r"])
    assert cr == pytest.approx(spec["formula_value"], rel=1e-12)
    assert abs(cr - spec["page_printed_value"]) > 0.5      # the printed figure is not the formula's
    pc = oracle.param_counts(d=4096, f=4096, E=8, G=1, r=16)
    # one matrix type of one group reproduces CR exactly
    assert pc["standard"] / pc["clustered"] == pytest.approx(cr, rel=1e-12)

