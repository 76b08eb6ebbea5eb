"""The compression step on the GPU (moe_hier_compress, moe_hier_quantise_int4) against its oracle.

Bars: the INT4 codes and FP16 scales of the quantiser bit-exact on the same FP32 input (the code is
decided in FP32 on both sides); the BF16 base bit-exact (same FP32 summation order); the truncated
SVD, which the GPU computes by a randomised range finder in FP32 and the oracle by an FP64 SVD:
the kept singular values within 1e-4 relative and the rank-r product B A^T within 1e-3 of the
oracle's in relative Frobenius norm; the reported reconstruction error equal to the oracle's
formula applied to the GPU's own codes (1e-6), and within 2e-3 (absolute) of the oracle's own
pipeline's error.
"""
import numpy as np
import pytest
import torch

from oracle import compress as C
import oracle
from synth import COMPRESS_CONFIGS, CompressConfig, make_dense_experts

pytestmark = pytest.mark.gpu

DIMS = {"gate": ("d", "f"), "up": ("d", "f"), "down": ("f", "d")}   # (d_in, d_out) attribute names


@pytest.fixture(scope="module")
def L(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    from compressed_expert_two_b300 import _lib
    return _lib


def run_gpu(L, cfg, inp, kind):
    d_in, d_out = (getattr(cfg, a) for a in DIMS[kind])
    E, G, r = cfg.E, cfg.G, cfg.r
    desc = L.MoeHierCompressDesc(E=E, G=G, d_out=d_out, d_in=d_in, rank=r, sketch=cfg.l,
                                 power_iters=cfg.power_iters)
    dev = "cuda"
    W = inp[kind]["W"].to(dev).contiguous()
    omega = inp[kind]["omega"].to(dev).contiguous()
    o = {"base": torch.empty(G, d_out, d_in, dtype=torch.bfloat16, device=dev),
         "Aq": torch.empty(E, r, d_in // 2, dtype=torch.uint8, device=dev),
         "As": torch.empty(E, r, d_in // 64, dtype=torch.float16, device=dev),
         "Bq": torch.empty(E, r, d_out // 2, dtype=torch.uint8, device=dev),
         "Bs": torch.empty(E, r, d_out // 64, dtype=torch.float16, device=dev),
         "sigma": torch.empty(E, r, dtype=torch.float32, device=dev),
         "err": torch.empty(E, dtype=torch.float64, device=dev),
         "At": torch.empty(E, r, d_in, dtype=torch.float32, device=dev),
         "Bt": torch.empty(E, r, d_out, dtype=torch.float32, device=dev)}
    nws = L.moe_hier_compress_workspace_size(desc)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    gm = inp["group_map"].to(torch.int32).contiguous()
    L.moe_hier_compress(desc, W, gm, omega, o["base"], o["Aq"], o["As"], o["Bq"], o["Bs"], o["sigma"], o["err"],
                        o["At"], o["Bt"], ws, nws, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in o.items()}


def test_quantiser_bit_exact(L, cuda_ok):
    rng = np.random.default_rng(9)
    v = (rng.standard_normal((40, 512)) * np.exp2(rng.uniform(-12, 4, (40, 1)))).astype(np.float32)
    v[3] = 0.0
    v[4, :64] = (np.arange(64) - 32) * (3.0 / 14.0)        # half-code ties at scale 3/7
    v[5, :64] = -v[5, :64]
    vd = torch.from_numpy(v).cuda()
    codes = torch.empty(40, 256, dtype=torch.uint8, device="cuda")
    scales = torch.empty(40, 8, dtype=torch.float16, device="cuda")
    L.moe_hier_quantise_int4(vd, 40, 512, codes, scales, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    q, s = C.quantise_int4_g64(v)
    assert np.array_equal(codes.cpu().numpy(), q)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), s.view(np.uint16))


@pytest.mark.parametrize("kind", ["gate", "down"])
def test_compress_small_layer_against_oracle(L, kind):
    cfg = CompressConfig("t", E=8, G=2, d=256, f=384, r=16, seed=21)
    inp = make_dense_experts(cfg, kinds=(kind,))
    got = run_gpu(L, cfg, inp, kind)
    W = inp[kind]["W"].float().numpy()
    gm = inp["group_map"].numpy()
    ref = C.compress_matrix(W, gm, cfg.G, cfg.r)
    assert np.array_equal(got["base"].float().numpy(), ref["base"])
    sig = got["sigma"].numpy().astype(np.float64)
    assert np.allclose(sig, ref["sigma"], rtol=1e-4, atol=0)
    for e in range(cfg.E):
        R = W[e].astype(np.float64) - ref["base"][gm[e]].astype(np.float64)
        B, A, _ = C.tsvd(R, cfg.r)
        want = B @ A.T
        have = got["Bt"][e].double().numpy().T @ got["At"][e].double().numpy()
        assert np.linalg.norm(have - want) <= 1e-3 * np.linalg.norm(want), e
        # balanced split, as the oracle's
        assert np.allclose(np.linalg.norm(got["At"][e].double().numpy(), axis=1), np.sqrt(sig[e]), rtol=2e-3)
        # the reported error is the oracle's formula on the GPU's own codes
        mine = C.reconstruction_error(W[e], ref["base"][gm[e]],
                                      oracle.dequant_int4(got["Aq"][e].numpy(), got["As"][e].numpy()),
                                      oracle.dequant_int4(got["Bq"][e].numpy(), got["Bs"][e].numpy()))
        assert abs(float(got["err"][e]) - mine) <= 1e-6
        assert abs(float(got["err"][e]) - ref["err"][e]) <= 2e-3
        # and the codes are the quantiser's codes of the GPU's own FP32 factors
        q, s = C.quantise_int4_g64(got["At"][e].numpy())
        assert np.array_equal(q, got["Aq"][e].numpy()) and np.array_equal(s, got["As"][e].numpy())


@pytest.mark.slow
def test_compress_small_workload_full_size(L):
    """The small workload's gate matrices (16 experts of 2816 x 1024): every expert against the
    oracle's FP64 truncated SVD."""
    cfg = COMPRESS_CONFIGS["compress_small"]
    inp = make_dense_experts(cfg, kinds=("gate",))
    got = run_gpu(L, cfg, inp, "gate")
    W = inp["gate"]["W"].float().numpy()
    gm = inp["group_map"].numpy()
    base = C.group_mean_base(W, gm, cfg.G)
    assert np.array_equal(got["base"].float().numpy(), base)
    for e in range(cfg.E):
        R = W[e].astype(np.float64) - base[gm[e]].astype(np.float64)
        B, A, S = C.tsvd(R, cfg.r)
        assert np.allclose(got["sigma"][e].double().numpy(), S, rtol=1e-4)
        have = got["Bt"][e].double().numpy().T @ got["At"][e].double().numpy()
        assert np.linalg.norm(have - B @ A.T) <= 1e-3 * np.linalg.norm(B @ A.T), e
