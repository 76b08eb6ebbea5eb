"""The workspace-free permutation entry point, for callers that cannot allocate device memory.

Some hosts own all device memory through their own pool and forbid any other allocation, and
some latency-critical loops may not pay an allocation's implicit synchronisation; neither can
hand the library a workspace.  moe_hier_permute_noalloc serves them from a fixed scratch array
inside the library.  These tests call it through the C ABI and check that it returns exactly
what moe_hier_permute returns and what the oracle's permutation returns, on calls in a row with
different layers (each call reuses the array the one before left behind).  Batches of at most
1024 tokens are permuted by a single-CTA kernel that needs no histogram scratch; larger ones use
the array.  The cases cover both sides of that limit (1024 and 1025 tokens) and the largest layer
the array accepts, 2 * ceil(T/256) * (E + G) = 65,536 entries exactly.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from synth import MoEConfig, make_inputs

KEYS = ("perm", "inv_pos", "expert_begin", "expert_count", "group_begin", "row_asg", "row_of", "row_begin")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from compressed_expert_two_b300 import _lib
    P = ctypes.c_void_p
    _lib.lib.moe_hier_permute_noalloc.argtypes = [ctypes.POINTER(_lib.MoeHierDesc)] + [P] * 11
    _lib.lib.moe_hier_permute_noalloc.restype = ctypes.c_int
    return _lib


def layer_case(**kw):
    base = dict(name="noalloc", T=5000, d=256, f=192, E=32, G=4, kg=2, ke=3, r=16, dtype="bf16",
                resid="int4", group_map="perm", seed=41)
    base.update(kw)
    return MoEConfig(**base)


def noalloc_permute(L, layer, eidx):
    cfg, T, dev = layer.cfg, layer.T, layer.device
    i32 = dict(dtype=torch.int32, device=dev)
    p = {"perm": torch.full((T * cfg.k,), -1, **i32), "inv_pos": torch.full((T * cfg.k,), -1, **i32),
         "expert_begin": torch.full((cfg.E,), -1, **i32), "expert_count": torch.full((cfg.E,), -1, **i32),
         "group_begin": torch.full((cfg.G + 1,), -1, **i32), "row_asg": torch.full((T * cfg.kg,), -1, **i32),
         "row_of": torch.full((T * cfg.kg,), -1, **i32), "row_begin": torch.full((cfg.G + 1,), -1, **i32)}
    rc = L.lib.moe_hier_permute_noalloc(ctypes.byref(layer.desc), layer.group_map.data_ptr(), eidx.data_ptr(),
                                        *[p[k].data_ptr() for k in KEYS], layer.stream)
    assert rc == L.MOE_OK, L.status_string(rc)
    return p


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute_twice(L, cuda_ok):
    from compressed_expert_two_b300.layer import DeviceLayer
    cases = [layer_case(), layer_case(T=8000, d=384, E=64, G=8, kg=2, ke=3, group_map="contiguous", seed=42,
                                      zipf_s=1.2),
             layer_case(T=1024, seed=43),                 # single-CTA kernel, no scratch
             layer_case(T=1025, seed=44),                 # smallest batch that uses the array
             # the largest layer the array holds: 2 * 256 blocks * (120 + 8) keys = 65,536 entries
             layer_case(T=65536, d=128, f=64, E=120, G=8, kg=1, ke=2, group_map="contiguous", seed=45)]
    for cfg in cases:
        inp = make_inputs(cfg)
        layer = DeviceLayer(inp, device="cuda")
        eidx = layer.route()["eidx"]
        want = layer.permute(eidx)
        got = noalloc_permute(L, layer, eidx)
        torch.cuda.synchronize()
        ref = oracle.permute(eidx.cpu().numpy(), inp["group_map"].numpy(), cfg.G, cfg.ke)
        for k in KEYS:
            assert torch.equal(got[k], want[k]), (cfg.name, cfg.T, k)
            assert np.array_equal(got[k].cpu().numpy(), ref[k]), (cfg.name, cfg.T, k)


def test_noalloc_rejects_layers_beyond_its_scratch(L):
    """2 * ceil(T/256) * (E + G) int32 must fit in the 65,536-entry array; checked on the host
    before anything touches the GPU."""
    desc = L.MoeHierDesc(T=1 << 20, d_model=128, d_ff=256, E=64, G=8, topk_group=1, topk_expert=2, rank=0,
                         act_dtype=L.MOE_BF16, resid_fmt=L.MOE_RESID_INT4_G64)
    gm = np.repeat(np.arange(8, dtype=np.int32), 8)
    fake = 1 << 20   # never dereferenced: the size check fails first
    rc = L.lib.moe_hier_permute_noalloc(ctypes.byref(desc), gm.ctypes.data, fake, fake, fake, fake, fake, fake,
                                        fake, fake, fake, None)
    assert rc == L.MOE_ERR_WORKSPACE
