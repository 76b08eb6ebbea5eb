"""A bounded device-side wait that runs out (failure detection without a GPU fault).

Every wait in the library's kernels is bounded; when one runs out the kernel writes
MOE_ERR_TIMEOUT to the workspace status word, leaves its loops and returns, so the context stays
usable and the host reads the condition with moe_hier_get_status.  The wait driven here is the
grid-wide barrier of the single-launch permutation (batches of more than 1024 tokens): the test
aid moe_hier_debug_set_wait makes it expect one arrival that nothing sends, with a 1 ms limit,
so every block gives up.  No kernel traps, faults or hangs; the next call, with the default
setting, must return outputs identical to the oracle's permutation.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import MoEConfig, make_inputs

pytestmark = pytest.mark.gpu

KEYS = ("perm", "inv_pos", "expert_begin", "expert_count", "group_begin", "row_asg", "row_of", "row_begin")


@pytest.fixture(scope="module")
def L(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    from compressed_expert_two_b300 import _lib
    return _lib


def test_permutation_wait_runs_out_then_the_next_call_is_exact(L):
    from compressed_expert_two_b300.layer import DeviceLayer
    cfg = MoEConfig("timeout", T=5000, d=256, f=192, E=32, G=4, kg=2, ke=3, r=16, dtype="bf16",
                    resid="int4", group_map="perm", seed=51)
    inp = make_inputs(cfg)
    layer = DeviceLayer(inp, device="cuda")
    eidx = layer.route()["eidx"]
    torch.cuda.synchronize()
    ref = oracle.permute(eidx.cpu().numpy(), inp["group_map"].numpy(), cfg.G, cfg.ke)

    layer.ws[:16].zero_()                                     # clear the status word
    L.moe_hier_debug_set_wait(1_000_000, 1)                   # 1 ms; one arrival that never comes
    try:
        layer.permute(eidx)
        st = L.moe_hier_get_status(layer.ws, layer.stream)
    finally:
        L.moe_hier_debug_set_wait(0, 0)
    assert st == L.MOE_ERR_TIMEOUT, L.status_string(st)
    word = layer.ws[:16].cpu().view(torch.int32)
    assert int(word[1]) == 90                                 # the permutation's barrier gave up
    torch.cuda.synchronize()                                  # no CUDA error on the stream

    layer.ws[:16].zero_()
    p = layer.permute(eidx)
    assert layer.status() == L.MOE_OK
    for k in KEYS:
        assert np.array_equal(p[k].cpu().numpy(), ref[k]), k


def test_wait_setting_rejects_negative_phantoms(L):
    with pytest.raises(L.MoeError):
        L.moe_hier_debug_set_wait(0, -1)
