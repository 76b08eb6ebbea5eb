"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: routing indices, gidx and every permutation output bit-exact; gates within 2e-5; layer
output y within max|y - y_ref| <= 2e-2 max|y_ref| and sum|y - y_ref| <= 5e-3 sum|y_ref|
(BF16 inputs, FP32 accumulation).

Gates: with at least 1024 BF16 tokens the router computes the logits on the tensor cores (an FP32
sum in another order than the canonical one), settles every decision the error bound allows and
recomputes the rest in the canonical order, so indices stay exact while the gates of verified
tokens come from logits that differ from the canonical ones by a few units of 2^-24 sum|x_i w_i|
(measured up to 3e-6 at d_model = 4096); a softmax moves by at most the largest change of its
inputs, and 2e-5 leaves a margin above that.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, MoEConfig, make_inputs, variant

pytestmark = pytest.mark.gpu

MAX_TOL, MEAN_TOL, GATE_TOL = 2e-2, 5e-3, 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()


def device_layer(inp):
    from compressed_expert_two_b300.layer import DeviceLayer
    return DeviceLayer(inp, device="cuda")


def check_y(y_gpu, y_ref, what=""):
    y = y_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(y - y_ref)
    scale = np.abs(y_ref).max()
    assert err.max() <= MAX_TOL * scale, f"{what} max err {err.max() / scale:.3g} of max|y|"
    assert err.sum() <= MEAN_TOL * np.abs(y_ref).sum(), f"{what} mean rel err {err.sum() / np.abs(y_ref).sum():.3g}"
    return err.max() / scale, err.sum() / np.abs(y_ref).sum()


def check_routing(out, ref):
    assert np.array_equal(out["gidx"].cpu().numpy(), ref["gidx"])
    assert np.array_equal(out["eidx"].cpu().numpy(), ref["eidx"])
    gate = out["gate"].cpu().numpy().astype(np.float64)
    assert np.abs(gate - ref["gate"]).max() <= GATE_TOL
    # the slots a reading does not pick carry exactly zero (picked ones are positive)
    assert np.array_equal(gate > 0, ref["active"])


def small(**kw):
    base = dict(name="case", T=300, d=256, f=192, E=8, G=2, kg=1, ke=2, r=16, dtype="bf16",
                resid="int4", group_map="perm", seed=21)
    base.update(kw)
    return MoEConfig(**base)


# ------------------------------------------------------------------ whole layer, small sizes
CASES = {
    "tiny_f32": CONFIGS["tiny_f32"],
    "tiny_f32_amp": variant(CONFIGS["tiny_f32"], "amplified"),
    "tiny_f32_base0": variant(CONFIGS["tiny_f32"], "base_zero"),
    "small_bf16_int4": CONFIGS["small_bf16_int4"],
    "bf16_ragged": small(),
    "bf16_amp": variant(small(seed=22), "amplified"),
    "bf16_base0": variant(small(seed=23), "base_zero"),
    "bf16_rank0": variant(small(seed=24), "rank0"),
    "bf16_kg2_ke3": small(T=515, E=32, G=4, kg=2, ke=3, f=320, group_map="contiguous", seed=25,
                          resid_std=0.2),
    "bf16_zipf": small(T=777, d=384, E=64, G=8, kg=2, ke=3, group_map="contiguous", seed=26,
                       zipf_s=1.2, resid_std=0.2),
    "bf16_one_token": small(T=1, seed=27),
    "bf16_rows2500_ke1": small(T=2500, d=512, f=384, ke=1, seed=38, resid_std=0.2),
    "bf16_rows2200_kg2": small(T=1100, d=512, f=256, E=16, G=4, kg=2, ke=2, seed=39, resid_std=0.2),
    "bf16_rows2200_krp128_ke3": small(T=1100, d=256, f=320, E=64, G=8, kg=2, ke=3, seed=43, resid_std=0.2,
                                      group_map="contiguous"),
    "bf16_rows2100_ke3": small(T=2100, d=256, f=192, E=16, G=4, kg=1, ke=3, seed=44, resid_std=0.2),
    "bf16_rows2100_ke4": small(T=2100, d=256, f=320, E=16, G=4, kg=1, ke=4, seed=45, resid_std=0.2),
    "bf16_fused_route_L8": small(T=1500, d=256, f=192, E=16, G=8, kg=2, ke=2, seed=46, resid_std=0.2),
    # tensor-core router, general selection path (more than 8 members, more than 8 groups)
    "bf16_tc_route_K16": small(T=1200, d=256, f=192, E=64, G=4, kg=2, ke=3, seed=48, resid_std=0.2),
    "bf16_tc_route_G16": small(T=1300, d=256, f=192, E=64, G=16, kg=3, ke=2, seed=49, resid_std=0.2),
    "bf16_K32": small(T=300, E=128, G=4, kg=2, ke=3, group_map="perm", seed=36, resid_std=0.2),
    "bf16_G64": small(T=200, E=128, G=64, kg=3, ke=2, group_map="perm", seed=37, resid_std=0.2),
    "bf16_K1": small(T=200, E=4, G=4, kg=2, ke=1, seed=28),
    "f32_kg2": small(T=130, dtype="f32", resid="f32", r=4, kg=2, ke=1, E=8, G=4, seed=29, resid_std=0.2),
    # the across-groups reading: top-k_e over the union of the chosen groups, zero gates elsewhere
    "bf16_across_kg2_ke3": small(T=1200, d=512, f=320, E=64, G=8, kg=2, ke=3, group_map="contiguous", seed=55,
                                 zipf_s=1.2, resid_std=0.2, route="across"),
    "bf16_across_few_tokens": small(T=300, E=32, G=4, kg=2, ke=2, seed=56, resid_std=0.2, route="across"),
    "f32_across": small(T=130, dtype="f32", resid="f32", r=4, kg=2, ke=2, E=12, G=3, seed=57, resid_std=0.2,
                        route="across"),
    # the descriptor's limits: 256 experts, 32 per group, 16 routed experts per token (2 x 8), rank 64
    "bf16_max_experts_k16": small(T=130, d=256, f=128, E=256, G=8, kg=2, ke=8, group_map="perm", seed=65,
                                  resid_std=0.2),
    "bf16_max_experts_k16_many_tokens": small(T=1100, d=256, f=128, E=256, G=8, kg=2, ke=8, group_map="contiguous",
                                            seed=66, resid_std=0.2),
    "f32_rank64": small(T=70, dtype="f32", resid="f32", r=64, kg=1, ke=2, E=8, G=2, seed=67, resid_std=0.05),
}


@pytest.mark.parametrize("name", list(CASES))
def test_forward_parity(name):
    cfg = CASES[name]
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    ref = oracle.forward(inp)
    check_routing(out, ref)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    check_y(out["y"], ref["y"], name)


def test_stages_match_oracle_and_forward():
    cfg = small(T=515, E=32, G=4, kg=2, ke=3, f=320, group_map="contiguous", seed=31)
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    ref = oracle.forward(inp)
    r = layer.route()
    check_routing(r, ref)
    p = layer.permute(r["eidx"])
    for key in ("perm", "inv_pos", "expert_begin", "expert_count", "group_begin", "row_asg",
                "row_of", "row_begin"):
        assert np.array_equal(p[key].cpu().numpy(), ref[key]), key
    y_rows = layer.ffn(layer.x, r["eidx"], r["gate"], p["row_asg"], p["row_begin"])
    y = layer.combine(y_rows)
    y_fwd = layer.forward()["y"]
    torch.cuda.synchronize()
    check_y(y, ref["y"], "stages")
    assert torch.equal(y, y_fwd)            # same kernels, same order: identical bits


def test_all_tokens_one_group_and_empty_experts():
    cfg = small(T=256, E=16, G=4, seed=33)
    inp = make_inputs(cfg)
    inp["b_group"] = torch.tensor([0.0, 0.0, 50.0, 0.0])    # every token picks group 2
    layer = device_layer(inp)
    out = layer.forward()
    ref = oracle.forward(inp)
    check_routing(out, ref)
    assert np.all(ref["gidx"] == 2)
    p = layer.permute(out["eidx"])
    for key in ("expert_begin", "expert_count", "group_begin", "row_begin"):
        assert np.array_equal(p[key].cpu().numpy(), ref[key]), key
    check_y(out["y"], ref["y"])


def route_redo(layer):
    """Tokens the tensor-core router left to the canonical-order kernels in the last call (a
    counter of the status word at the start of the workspace)."""
    return int(layer.ws[12:16].view(torch.int32).item())


@pytest.mark.parametrize("kind", ["group_rows", "expert_rows", "zero_tokens"])
def test_tc_router_ties(kind):
    """Exact ties (duplicated router rows, all-zero tokens) cannot be settled from the tensor-core
    logits: those tokens go through the canonical order and the indices still equal the oracle's
    (ties -> lower index)."""
    cfg = small(T=2048, d=512, f=192, E=32, G=4, kg=2, ke=2, group_map="contiguous", seed=52, resid_std=0.2)
    inp = make_inputs(cfg)
    if kind == "group_rows":
        inp["w_group"][1] = inp["w_group"][0]
    elif kind == "expert_rows":
        inp["w_expert"][3] = inp["w_expert"][5]
    else:
        inp["x"][::5] = 0
    layer = device_layer(inp)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    redo = route_redo(layer)
    ref = oracle.forward(inp)
    check_routing(out, ref)
    assert np.array_equal(out["perm"].cpu().numpy(), ref["perm"])
    check_y(out["y"], ref["y"], kind)
    assert 0 < redo < cfg.T
    if kind == "zero_tokens":
        assert redo >= (cfg.T + 4) // 5


@pytest.mark.parametrize("many", [True, False])
def test_recomputed_logits_are_canonical_bits(many):
    """The canonical-order kernel's logits of the tokens the tensor-core router left over equal the
    oracle's FP32 canonical logits bit for bit (read from the workspace: status word, then the
    [T][G+E] logits scratch, then the [T] token list, each region 256-byte aligned).  Many listed
    tokens take the 8-token tiles, few the one-token-per-warp form."""
    cfg = small(T=2048, d=512, f=192, E=32, G=4, kg=2, ke=2, group_map="contiguous", seed=54, resid_std=0.2)
    inp = make_inputs(cfg)
    if many:
        inp["w_group"][2] = inp["w_group"][1]               # exact ties for most tokens
    else:
        inp["w_expert"][9] = inp["w_expert"][10]            # ties for the tokens that reach them
    layer = device_layer(inp)
    layer.route()
    torch.cuda.synchronize()
    n = route_redo(layer)
    R = cfg.G + cfg.E
    nw = 148 * 8                                            # warps of the recompute launch
    if many:
        assert n * ((R + 7) // 8) > 2 * nw
    else:
        assert 0 < n and n * ((R + 7) // 8) <= 2 * nw
    off_logits = 256
    off_redo = off_logits + (cfg.T * R * 4 + 255) // 256 * 256
    toks = layer.ws[off_redo:off_redo + 4 * n].view(torch.int32).cpu().numpy()
    got = layer.ws[off_logits:off_logits + 4 * n * R].view(torch.float32).cpu().numpy().reshape(n, R)
    assert len(set(toks.tolist())) == n and toks.min() >= 0 and toks.max() < cfg.T
    x = oracle.moe._np(inp["x"])[toks]
    want = np.concatenate([oracle.canonical_logits(x, oracle.moe._np(inp["w_group"])),
                           oracle.canonical_logits(x, oracle.moe._np(inp["w_expert"]))], axis=1)
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))


def test_tc_router_standalone_route_call():
    """moe_hier_route on its own (no forward before it) clears the recompute counter itself."""
    cfg = small(T=1536, d=256, E=32, G=4, kg=1, ke=2, seed=53)
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    ref = oracle.forward(inp)
    for _ in range(3):
        r = layer.route()
        torch.cuda.synchronize()
        check_routing(r, ref)
        assert route_redo(layer) < cfg.T // 4


def synthetic_eidx(T, group_map, G, kg, ke, seed, skew=0.0):
    """Seeded routing decisions: kg distinct groups per token (weights ~ (g+1)^-skew), then ke
    distinct experts of each chosen group."""
    rng = np.random.default_rng(seed)
    members = [np.flatnonzero(group_map == g) for g in range(G)]
    w = (np.arange(G) + 1.0) ** -skew
    w /= w.sum()
    eidx = np.empty((T, kg * ke), dtype=np.int32)
    for t in range(T):
        gs = rng.choice(G, size=kg, replace=False, p=w)
        for j, g in enumerate(gs):
            eidx[t, j * ke:(j + 1) * ke] = rng.choice(members[g], size=ke, replace=False)
    return eidx


@pytest.mark.parametrize("T,E,G,kg,ke,skew", [(20, 64, 8, 2, 3, 0.0), (64, 32, 8, 1, 2, 0.0),
                                              (1000, 256, 8, 2, 4, 1.0), (1024, 16, 4, 1, 2, 0.0),
                                              (1025, 16, 4, 1, 2, 0.0), (3000, 64, 8, 2, 3, 1.2),
                                              (9000, 8, 2, 1, 2, 0.0), (16384, 64, 8, 2, 3, 2.5)])
def test_permute_batches(T, E, G, kg, ke, skew):
    """One-CTA batches (up to 1024 tokens, down to a single warp) and multi-block batches, called
    twice in a row through the stand-alone entry point: every output bit-exact both times."""
    cfg = small(T=T, E=E, G=G, kg=kg, ke=ke, seed=40 + T % 97)
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    gm = inp["group_map"].numpy()
    eidx = synthetic_eidx(T, gm, G, kg, ke, seed=T, skew=skew)
    ref = oracle.permute(eidx, gm, G, ke)
    e_dev = torch.from_numpy(eidx).cuda()
    for _ in range(2):
        p = layer.permute(e_dev)
        torch.cuda.synchronize()
        assert layer.status() == 0
        for key, want in ref.items():
            assert np.array_equal(p[key].cpu().numpy(), want), key


def test_empty_batch():
    cfg = small(T=0, seed=34)
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    out = layer.forward()
    p = layer.permute(out["eidx"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert p["row_begin"].cpu().tolist() == [0] * (cfg.G + 1)


def test_repeat_calls_are_deterministic():
    inp = make_inputs(small(T=400, seed=35))
    layer = device_layer(inp)
    a = layer.forward()
    b = layer.forward()
    torch.cuda.synchronize()
    for k in ("y", "eidx", "gate", "perm"):
        assert torch.equal(a[k], b[k]), k


# ------------------------------------------------------------------ the full-size workloads
def full_size_check(name, n_sample, cfg=None):
    cfg = cfg or CONFIGS[name]
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    out = layer.forward()
    torch.cuda.synchronize()
    assert layer.status() == 0
    gm = inp["group_map"].numpy()
    routing = oracle.route(oracle.moe._np(inp["x"]), oracle.moe._np(inp["w_group"]),
                           oracle.moe._np(inp["b_group"]), oracle.moe._np(inp["w_expert"]), gm,
                           cfg.kg, cfg.ke, cfg.route)
    check_routing(out, routing)
    pref = oracle.permute(routing["eidx"], gm, cfg.G, cfg.ke)
    assert np.array_equal(out["perm"].cpu().numpy(), pref["perm"])
    rng = np.random.default_rng(cfg.seed)
    toks = np.sort(rng.choice(cfg.T, size=min(n_sample, cfg.T), replace=False))
    toks[0], toks[-1] = 0, cfg.T - 1
    y_ref, _ = oracle.forward_tokens(inp, toks, routing=routing)
    check_y(out["y"][torch.from_numpy(toks).cuda()], y_ref, name)


@pytest.mark.slow
@pytest.mark.parametrize("name,n", [("mixtral_prefill", 24), ("finegrained_skewed", 64), ("decode", 8),
                                    ("finegrained_across", 64)])
def test_full_size_sampled(name, n):
    full_size_check(name, n)


@pytest.mark.parametrize("T,ke,seed", [(2304, 2, 41), (2100, 1, 42)])
def test_long_k_gate_up_sampled(T, ke, seed):
    """d_model = 4096 with more than 2048 rows: the CTA-pair double-buffered gate/up kernel, with
    a ragged last pair (T not a multiple of 256 rows per group); sampled tokens against the oracle."""
    cfg = small(T=T, d=4096, f=1024, E=8, G=2, kg=1, ke=ke, seed=seed, resid_std=0.2)
    full_size_check("long_k", 40, cfg)


@pytest.mark.parametrize("T,kg,ke,seed", [(1100, 2, 3, 61), (2100, 1, 3, 62), (2100, 1, 2, 63), (2300, 1, 1, 64)])
def test_wide_residual_many_rows_sampled(T, kg, ke, seed):
    """d_model = 2048 with 8 experts of rank 16 per group (a 128-column residual) and more than
    2048 rows: the persistent 128-column gate/up kernel over many items with one to three slots,
    ragged groups; sampled tokens against the oracle."""
    cfg = small(T=T, d=2048, f=384, E=32, G=4, kg=kg, ke=ke, seed=seed, resid_std=0.2)
    full_size_check("wide_residual", 48, cfg)


@pytest.mark.parametrize("T,ke,seed", [(6100, 2, 71), (6100, 1, 72)])
def test_pair_gate_up_many_items_sampled(T, ke, seed):
    """d_model = 4096 with about 6000 rows in two groups: the persistent CTA-pair gate/up kernel
    walks more (pair tile, chunk) items than there are clusters, so clusters take several items
    each (the stage ring, accumulator parity and slot phases carried across items), with ragged
    pair tiles; sampled tokens against the oracle."""
    cfg = small(T=T, d=4096, f=1024, E=8, G=2, kg=1, ke=ke, seed=seed, resid_std=0.2)
    full_size_check("pair_items", 48, cfg)


def test_pair_gate_up_skewed_groups_sampled():
    """The persistent CTA-pair gate/up kernel (d_model = 4096) under a Zipf(2.5) group load: one
    group holds most rows, the others a few ragged pair tiles or none; sampled tokens against
    the oracle."""
    cfg = small(T=4096, d=4096, f=1024, E=16, G=4, kg=1, ke=2, seed=75, resid_std=0.2, zipf_s=2.5,
                group_map="contiguous")
    full_size_check("pair_skewed", 48, cfg)


def test_persistent_down_gemm_sampled():
    """Many waves of down-projection tiles with a short K loop (d_ff = 256): the persistent grouped
    GEMM with double-buffered accumulators; sampled tokens against the oracle, ragged groups."""
    cfg = small(T=16384, d=1024, f=256, E=8, G=2, kg=1, ke=2, seed=47, resid_std=0.2)
    full_size_check("persist", 48, cfg)


@pytest.mark.parametrize("name", ["bf16_ragged", "bf16_kg2_ke3", "bf16_rows2500_ke1", "small_bf16_int4",
                                  "bf16_rows2200_krp128_ke3", "bf16_one_token"])
def test_prepared_stacks_forward_is_identical(name):
    """moe_hier_forward_prepared (residual stacks built once by moe_hier_prepare) returns exactly
    what moe_hier_forward returns, twice in a row (the stacks are not consumed)."""
    inp = make_inputs(CASES[name])
    layer = device_layer(inp)
    want = layer.forward()
    layer.prepare()
    for _ in range(2):
        got = layer.forward_prepared()
        torch.cuda.synchronize()
        assert layer.status() == 0
        for k in ("y", "gidx", "eidx", "gate", "perm"):
            assert torch.equal(got[k], want[k]), k


def test_prepared_stacks_decode_shape_sampled():
    """A decode-shaped layer (64 tokens, d_model 4096) through the prepared path against the oracle."""
    cfg = small(T=64, d=4096, f=1024, E=32, G=8, kg=1, ke=2, seed=58, resid_std=0.2, group_map="contiguous")
    inp = make_inputs(cfg)
    layer = device_layer(inp).prepare()
    out = layer.forward_prepared()
    torch.cuda.synchronize()
    ref = oracle.forward(inp)
    check_routing(out, ref)
    check_y(out["y"], ref["y"], "prepared decode")


@pytest.mark.parametrize("kw", [dict(T=64, d=512, f=256, E=32, G=8, kg=1, ke=2, seed=61),
                                dict(T=200, d=256, f=192, E=64, G=8, kg=2, ke=3, seed=62, group_map="contiguous"),
                                dict(T=129, d=256, f=192, E=64, G=16, kg=2, ke=2, seed=63),
                                dict(T=256, d=384, f=128, E=16, G=4, kg=1, ke=2, seed=64, zipf_s=1.2)])
def test_small_batches_forward_matches_stages_and_oracle(kw):
    """Batches of at most 256 tokens (the decode shapes): moe_hier_forward and the stage-by-stage
    calls (route, permute, ffn, combine) give the same routing, permutation and output bit for
    bit, and both match the oracle."""
    cfg = small(resid_std=0.2, **kw)
    inp = make_inputs(cfg)
    layer = device_layer(inp)
    fwd = layer.forward()
    r = layer.route()
    pm = layer.permute(r["eidx"])
    y = layer.combine(layer.ffn(layer.x, r["eidx"], r["gate"], pm["row_asg"], pm["row_begin"]))
    torch.cuda.synchronize()
    assert layer.status() == 0
    for k in ("gidx", "eidx", "gate"):
        assert torch.equal(fwd[k], r[k]), k
    assert torch.equal(fwd["perm"], pm["perm"])
    assert torch.equal(fwd["y"], y)
    ref = oracle.forward(inp)
    check_routing(fwd, ref)
    assert np.array_equal(fwd["perm"].cpu().numpy(), ref["perm"])
    check_y(fwd["y"], ref["y"], "small batch")
