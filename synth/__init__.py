"""Seeded synthetic inputs for the clustered, compressed MoE layer.

This module is shared by the CPU oracle (under ``oracle/``, test infrastructure) and by the CUDA
path (tests and ``bench.py``).  It holds none of the layer's arithmetic: it only draws tensors in a
fixed order from a seeded torch CPU generator and stores them in the formats the layer consumes.

Formats (all row-major, ``nn.Linear`` convention ``y = W x`` with ``W`` of shape [d_out][d_in]):

* ``x``         [T][d]          activations (BF16, or FP32 for the FP32 configuration)
* ``w_group``   [G][d]          group router rows;  ``w_expert`` [E][d] expert router rows
* ``b_group``   [G] FP32 or None  additive group-router bias (the skewed configuration only)
* ``group_map`` [E] int32       group of each expert; exactly K = E/G experts per group
* ``w_gate``, ``w_up`` [G][f][d];  ``w_down`` [G][d][f]   per-group shared base matrices
* residual factors of expert i for matrix m in (gate, up, down), for W~ = W_base + B A^T with
  A in R^{d_in x r}, B in R^{d_out x r} ("Breaking the MoE LLM Trilemma", key design 2, W~ eq.):
  stored rank-major, i.e. as A^T [E][r][d_in] and B^T [E][r][d_out].
  - FP32 format: plain float32 tensors.
  - INT4 group-64 format: symmetric 4-bit codes packed two per byte along the feature axis,
    element 2j in the HIGH nibble and element 2j+1 in the LOW nibble of byte j, stored as the
    unsigned nibble u = q + 8 (q in [-7, 7]), so value = (u - 8) * scale; one FP16 scale per 64
    consecutive elements of a rank row ([E][r][d/64]).  The nibble order and zero point follow
    the INT4 unpack convention printed on the MoE-whitepaper page (section 3.2, fused FP8xINT4
    kernel listing).  Producing the codes is the offline compression step; the forward pass only
    consumes them, and the dequantised values are the truth.

Synthetic recipe (seeded ``torch.Generator().manual_seed(seed)``; draw order x, w_group, b_group,
w_expert, group-map permutation, w_gate, w_up, w_down, then (A, B) for gate, up, down):
x ~ N(0,1); base W ~ N(0, 1/d_in); routers ~ N(0, 1/d); A, B ~ N(0, resid_std^2).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch

QGROUP = 64  # elements per INT4 scale group


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int          # d_model
    f: int          # d_ff
    E: int
    G: int
    kg: int         # top-k groups
    ke: int         # top-k experts inside each chosen group
    r: int          # residual rank
    dtype: str      # "f32" or "bf16": x, routers, base weights, y
    resid: str      # "f32" or "int4"
    group_map: str  # "contiguous" or "perm"
    seed: int
    zipf_s: Optional[float] = None   # group-router bias so group load follows Zipf(s)
    resid_std: float = 0.02
    base_scale: float = 1.0          # 0.0 gives the base-zero (pure low-rank) variant
    route: str = "within"            # "within": top-ke in each chosen group; "across": top-ke over their union

    @property
    def K(self) -> int:
        return self.E // self.G

    @property
    def k(self) -> int:
        return self.kg * self.ke

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# The five workloads the layer is measured on (Mixtral-shaped and fine-grained shapes as stated).
CONFIGS: Dict[str, MoEConfig] = {
    "tiny_f32": MoEConfig("tiny_f32", T=256, d=128, f=256, E=8, G=2, kg=1, ke=2, r=4,
                          dtype="f32", resid="f32", group_map="contiguous", seed=0),
    "small_bf16_int4": MoEConfig("small_bf16_int4", T=4096, d=1024, f=2816, E=16, G=4, kg=1, ke=2,
                                 r=16, dtype="bf16", resid="int4", group_map="perm", seed=1),
    "mixtral_prefill": MoEConfig("mixtral_prefill", T=8192, d=4096, f=14336, E=8, G=2, kg=1, ke=2,
                                 r=16, dtype="bf16", resid="int4", group_map="contiguous", seed=2),
    "finegrained_skewed": MoEConfig("finegrained_skewed", T=16384, d=2048, f=1408, E=64, G=8, kg=2,
                                    ke=3, r=16, dtype="bf16", resid="int4", group_map="contiguous",
                                    seed=3, zipf_s=1.2),
    "decode": MoEConfig("decode", T=64, d=4096, f=14336, E=32, G=8, kg=1, ke=2, r=16,
                        dtype="bf16", resid="int4", group_map="contiguous", seed=4),
}
CONFIG_ORDER = ["tiny_f32", "small_bf16_int4", "mixtral_prefill", "finegrained_skewed", "decode"]
# Decode with 4 tokens per step and skewed group loads: most groups sit idle in any one step,
# the case the idle-group offload serves (bases of 4 of the 8 groups cached on the device).
CONFIGS["decode_offload"] = MoEConfig("decode_offload", T=4, d=4096, f=14336, E=32, G=8, kg=1, ke=2, r=16,
                                      dtype="bf16", resid="int4", group_map="contiguous", seed=4, zipf_s=1.2)
# The other reading of the fine-grained workload: top-3 experts over the union of the 2 chosen groups.
CONFIGS["finegrained_across"] = CONFIGS["finegrained_skewed"].replace(name="finegrained_across", route="across")


def _torch_dtype(cfg: MoEConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def pack_int4_g64(w: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Store float rank rows w [..., n] (n % 64 == 0) in the INT4 group-64 format.

    scale = fp16(absmax/7) per 64 elements; code q = clamp(round_half_even(w/scale), -7, 7);
    nibble u = q + 8; element 2j -> high nibble of byte j, 2j+1 -> low nibble.
    Returns (packed uint8 [..., n/2], scales fp16 [..., n/64]).
    """
    n = w.shape[-1]
    assert n % QGROUP == 0
    wg = w.float().reshape(*w.shape[:-1], n // QGROUP, QGROUP)
    amax = wg.abs().amax(dim=-1)
    scale16 = (amax / 7.0).to(torch.float16)
    s = scale16.float().unsqueeze(-1)
    q = torch.where(s > 0, torch.round(wg / torch.where(s > 0, s, torch.ones_like(s))),
                    torch.zeros_like(wg)).clamp_(-7, 7)
    u = (q + 8).to(torch.uint8).reshape(*w.shape[:-1], n)
    packed = (u[..., 0::2] << 4) | u[..., 1::2]
    return packed.contiguous(), scale16.contiguous()


def _group_map(cfg: MoEConfig, gen: torch.Generator) -> torch.Tensor:
    if cfg.group_map == "contiguous":
        return (torch.arange(cfg.E) // cfg.K).to(torch.int32)
    perm = torch.randperm(cfg.E, generator=gen)
    return (perm // cfg.K).to(torch.int32)


def _zipf_bias(cfg: MoEConfig, gen: torch.Generator) -> torch.Tensor:
    """b_g = ln p_{pi(g)}, p_j proportional to j^-s (j = 1..G), pi a seeded permutation."""
    j = torch.arange(1, cfg.G + 1, dtype=torch.float64)
    p = j.pow(-cfg.zipf_s)
    p = p / p.sum()
    pi = torch.randperm(cfg.G, generator=gen)
    return torch.log(p[pi]).to(torch.float32)


def make_inputs(cfg: MoEConfig) -> dict:
    """Draw every input of the layer for ``cfg`` (CPU tensors)."""
    gen = torch.Generator().manual_seed(cfg.seed)
    dt = _torch_dtype(cfg)
    T, d, f, E, G, r = cfg.T, cfg.d, cfg.f, cfg.E, cfg.G, cfg.r

    def normal(shape, std):
        return torch.randn(*shape, generator=gen, dtype=torch.float32).mul_(std)

    out: dict = {"cfg": cfg}
    out["x"] = normal((T, d), 1.0).to(dt)
    out["w_group"] = normal((G, d), 1.0 / math.sqrt(d)).to(dt)
    out["b_group"] = _zipf_bias(cfg, gen) if cfg.zipf_s is not None else None
    out["w_expert"] = normal((E, d), 1.0 / math.sqrt(d)).to(dt)
    out["group_map"] = _group_map(cfg, gen)

    def base(shape, d_in):
        # Drawn one group at a time to bound host memory on the large shapes.
        t = torch.empty(shape, dtype=dt)
        for g in range(shape[0]):
            t[g] = normal(shape[1:], cfg.base_scale / math.sqrt(d_in)).to(dt)
        return t

    out["w_gate"] = base((G, f, d), d)
    out["w_up"] = base((G, f, d), d)
    out["w_down"] = base((G, d, f), f)

    dims = {"gate": (d, f), "up": (d, f), "down": (f, d)}   # (d_in, d_out)
    resid = {}
    for m in ("gate", "up", "down"):
        d_in, d_out = dims[m]
        At = normal((E, r, d_in), cfg.resid_std)     # A^T, rank-major
        Bt = normal((E, r, d_out), cfg.resid_std)    # B^T, rank-major
        if cfg.resid == "f32":
            resid[m] = {"A": At.contiguous(), "B": Bt.contiguous()}
        else:
            Aq, As = pack_int4_g64(At)
            Bq, Bs = pack_int4_g64(Bt)
            resid[m] = {"Aq": Aq, "As": As, "Bq": Bq, "Bs": Bs}
    out["resid"] = resid
    return out


def variant(cfg: MoEConfig, kind: str) -> MoEConfig:
    """Test variants that make every fused term visible above the float tolerance."""
    if kind == "amplified":
        return cfg.replace(name=cfg.name + "+amp", resid_std=0.2)
    if kind == "base_zero":
        return cfg.replace(name=cfg.name + "+base0", base_scale=0.0, resid_std=0.2)
    if kind == "rank0":
        return cfg.replace(name=cfg.name + "+r0", r=0)
    raise ValueError(kind)


# --------------------------------------------------------------------------------------------
# Dense experts for the compression step (the step that produces the layer's weights)
# --------------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class CompressConfig:
    name: str
    E: int
    G: int
    d: int          # d_model
    f: int          # d_ff
    r: int          # residual rank kept
    seed: int
    oversample: int = 16      # extra columns of the randomised range finder's test matrix
    power_iters: int = 4      # subspace iterations of the randomised range finder
    dev_scale: float = 0.05   # ||expert's own rank-r deviation||_F / ||shared part||_F
    noise: float = 0.01       # ||full-rank noise||_F / ||shared part||_F
    group_map: str = "contiguous"

    @property
    def K(self) -> int:
        return self.E // self.G

    @property
    def l(self) -> int:
        return self.r + self.oversample


COMPRESS_CONFIGS: Dict[str, CompressConfig] = {
    # the layer shapes of the small BF16 and Mixtral-shaped workloads, as dense experts
    "compress_small": CompressConfig("compress_small", E=16, G=4, d=1024, f=2816, r=16, seed=11),
    "compress_mixtral": CompressConfig("compress_mixtral", E=8, G=2, d=4096, f=14336, r=16, seed=12),
}


def make_dense_experts(cfg: CompressConfig, kinds=("gate", "up", "down")) -> dict:
    """Seeded dense expert weights W_i = shared_g + dev_i + noise_i, stored as BF16 [E][d_out][d_in]
    per matrix kind, with shared_g ~ N(0, 1/d_in) per group, dev_i = U_i V_i^T of rank r (Gaussian
    factors, scaled to dev_scale of the shared part's Frobenius norm) and Gaussian noise (noise of
    it): experts of a group that share most of their weights, each with a low-rank individuality.
    Also draws, per kind, the randomised range finder's Gaussian test matrix omega [d_in][r + p]
    (FP32): the random numbers the GPU's truncated SVD uses are inputs, not drawn on the device."""
    gen = torch.Generator().manual_seed(cfg.seed)
    dims = {"gate": (cfg.d, cfg.f), "up": (cfg.d, cfg.f), "down": (cfg.f, cfg.d)}   # (d_in, d_out)
    if cfg.group_map == "contiguous":
        gm = (torch.arange(cfg.E) // cfg.K).to(torch.int32)
    else:
        gm = (torch.randperm(cfg.E, generator=gen) // cfg.K).to(torch.int32)
    out = {"cfg": cfg, "group_map": gm}
    for m in kinds:
        d_in, d_out = dims[m]
        W = torch.empty(cfg.E, d_out, d_in, dtype=torch.bfloat16)
        for g in range(cfg.G):
            shared = torch.randn(d_out, d_in, generator=gen) / math.sqrt(d_in)
            for e in torch.nonzero(gm == g).flatten().tolist():
                U = torch.randn(d_out, cfg.r, generator=gen)
                V = torch.randn(d_in, cfg.r, generator=gen)
                dev = (U @ V.T) * (cfg.dev_scale / math.sqrt(d_in * cfg.r))
                noise = torch.randn(d_out, d_in, generator=gen) * (cfg.noise / math.sqrt(d_in))
                W[e] = (shared + dev + noise).to(torch.bfloat16)
        out[m] = {"W": W, "omega": torch.randn(d_in, cfg.l, generator=gen)}
    return out
