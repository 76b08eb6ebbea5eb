"""The tensor-core router's error bound, measured on the hardware.

The router accepts a token's decision from its tensor-core logits only when every pick's interval
[s_tc - delta, s_tc + delta] clears its competitors', with
    delta = c(d) ||x|| ||w|| + 2^-22 |s_tc|,  c(d) = 1.01 ((d/8 + 8) 2^-22 + (d/32 + 6) 2^-24).
The routing indices equal the canonical FP32 ones ("router in FP32", routing-mechanisms page
section 3.1) only if |s_tc - s_canonical| <= delta holds for every logit.  The test aid
moe_hier_debug_route_tc returns each token's tensor-core logits and deltas; this checks the
inequality element by element against the oracle's canonical logits, and the tensor-core share
of it, 1.01 (d/8 + 8) 2^-22 ||x|| ||w||, against the exact FP64 dot product, at d_model 256, 2048
and 4096, on Gaussian tokens and on adversarial ones: tokens scaled by 1e3, a wide spread of
exponents inside a row, heavy cancellation, an all-positive router row, and tokens equal to a
router row whose later products sit just below the accumulator's last bit (the worst case of a
tensor core that aligns and truncates products without guard bits).  The largest fractions used
are printed.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    from compressed_expert_two_b300 import _lib
    return _lib


def bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def adversarial_inputs(d: int, seed: int):
    cfg = MoEConfig("tc_bound", T=1024, d=d, f=128, E=64, G=8, kg=2, ke=3, r=16, dtype="bf16",
                    resid="int4", group_map="contiguous", seed=seed, zipf_s=1.2)
    inp = make_inputs(cfg)
    rng = np.random.default_rng(seed)
    x = inp["x"].float().numpy().copy()
    we = inp["w_expert"].float().numpy().copy()
    x[0:8] *= 1e3                                                     # large tokens
    spread = rng.standard_normal((8, d)) * np.exp2(rng.uniform(-20, 20, (8, d)))
    x[8:16] = spread                                                  # exponents across 40 binades
    half = rng.standard_normal((8, d // 2))
    x[16:24] = np.concatenate([half, -half * (1 + 2.0 ** -8)], axis=1)  # heavy cancellation
    we[1] = np.abs(we[1])                                             # all-positive router row
    x[24:32] = np.abs(x[24:32])                                       # ... and all-positive tokens
    # a router row that the alignment model loses most on, and tokens equal to it
    drop = np.full(d, math.sqrt(0.97 * 16 * 64 * 2.0 ** -23), dtype=np.float32)
    drop[:16] = 8.0
    we[5] = drop
    x[32:40] = drop
    drop4 = drop.copy()
    drop4[:64] = 8.0
    we[9] = drop4
    x[40:48] = drop4
    inp["x"] = torch.from_numpy(bf16(x)).to(torch.bfloat16)
    inp["w_expert"] = torch.from_numpy(bf16(we)).to(torch.bfloat16)
    return cfg, inp


@pytest.mark.parametrize("d", [256, 2048, 4096])
def test_tensor_core_logits_within_the_verification_bound(L, d):
    from compressed_expert_two_b300.layer import DeviceLayer
    cfg, inp = adversarial_inputs(d, seed=60 + d // 256)
    layer = DeviceLayer(inp, device="cuda")
    G, E = cfg.G, cfg.E
    out = torch.zeros(cfg.T, 2 * (G + E), dtype=torch.float32, device="cuda")
    L.moe_hier_debug_route_tc(layer.desc, layer.x, layer.w_group, layer.b_group, layer.w_expert,
                              layer.group_map, out, layer.ws, layer.ws_bytes, layer.stream)
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64)
    s_tc, delta = o[:, :G + E], o[:, G + E:]

    x = inp["x"].float().numpy()
    wg, we = inp["w_group"].float().numpy(), inp["w_expert"].float().numpy()
    bg = inp["b_group"].numpy() if inp["b_group"] is not None else None
    canon = np.concatenate([oracle.canonical_logits(x, wg, bg), oracle.canonical_logits(x, we)], axis=1)
    frac = np.abs(s_tc - canon.astype(np.float64)) / delta
    assert np.all(np.isfinite(frac))
    worst = np.unravel_index(np.argmax(frac), frac.shape)
    # the tensor-core share of the bound against the exact dot product (expert columns: no bias)
    x64, we64 = x.astype(np.float64), we.astype(np.float64)
    exact = x64 @ we64.T
    share = 1.01 * (d / 8 + 8) * 2.0 ** -22 * np.linalg.norm(x64, axis=1)[:, None] * \
        np.linalg.norm(we64, axis=1)[None, :]
    frac_tc = np.abs(s_tc[:, G:] - exact) / share
    print(f"d={d}: largest |s_tc - s_canonical| / delta = {frac.max():.4f} at token {worst[0]} column "
          f"{worst[1]}; largest |s_tc - exact| / tensor-core share = {frac_tc.max():.4f}")
    assert frac.max() <= 1.0
    assert frac_tc.max() <= 1.0
