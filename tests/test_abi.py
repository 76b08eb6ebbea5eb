"""C-ABI checks that need no GPU: the library loads, exports what the header declares, and
rejects bad arguments on the host before anything is enqueued."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from compressed_expert_two_b300 import _lib
    return _lib


def header_functions():
    src = open(os.path.join(ROOT, "include", "moehier.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_hier_\w+)\s*\(", src)))


def test_exports_match_header(L):
    names = header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L.lib, n), n
    assert sorted(L.EXPORTS) == sorted(n for n in names if n in L.EXPORTS)


def desc_for(L, **kw):
    base = dict(T=256, d_model=128, d_ff=256, E=8, G=2, topk_group=1, topk_expert=2, rank=4,
                act_dtype=L.MOE_F32, resid_fmt=L.MOE_RESID_F32)
    base.update(kw)
    return L.MoeHierDesc(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(E=9), -1), (dict(G=3, E=8), -1), (dict(topk_group=3), -1), (dict(topk_expert=5), -1),
    (dict(d_model=96), -1), (dict(d_ff=100), -1), (dict(rank=-1), -1), (dict(T=-1), -1),
    (dict(act_dtype=7), -1), (dict(resid_fmt=1), -2), (dict(rank=65), -2),
    (dict(E=512, G=2), -1), (dict(E=64, G=1, topk_expert=2), -2),
])
def test_invalid_descriptors(L, kw, code):
    st = ctypes.c_int(0)
    n = L.lib.moe_hier_workspace_size(ctypes.byref(desc_for(L, **kw)), ctypes.byref(st))
    assert n == 0 and st.value == code


def test_workspace_size_grows_with_T(L):
    a = L.moe_hier_workspace_size(desc_for(L, T=256))
    b = L.moe_hier_workspace_size(desc_for(L, T=512))
    assert 0 < a < b and a % 256 == 0


def test_bad_group_map_and_workspace_rejected_before_launch(L):
    import numpy as np
    d = desc_for(L)
    gm_bad = np.array([0, 0, 0, 0, 0, 1, 1, 1], dtype=np.int32)   # 5 experts in group 0
    fake = 1 << 20  # never dereferenced: validation fails first
    rc = L.lib.moe_hier_route(ctypes.byref(d), fake, fake, None, fake,
                              gm_bad.ctypes.data, fake, fake, fake, fake, 1 << 30, None)
    assert rc == L.MOE_ERR_INVALID
    gm = np.array([0, 0, 0, 0, 1, 1, 1, 1], dtype=np.int32)
    rc = L.lib.moe_hier_route(ctypes.byref(d), fake, fake, None, fake, gm.ctypes.data, fake, fake,
                              fake, fake, 16, None)
    assert rc == L.MOE_ERR_WORKSPACE
    rc = L.lib.moe_hier_route(ctypes.byref(d), fake, fake, None, fake, gm.ctypes.data, fake, fake,
                              fake, fake + 8, 1 << 30, None)
    assert rc == L.MOE_ERR_WORKSPACE                                   # misaligned
    rc = L.lib.moe_hier_route(ctypes.byref(d), None, fake, None, fake, gm.ctypes.data, fake, fake,
                              fake, fake, 1 << 30, None)
    assert rc == L.MOE_ERR_INVALID                                     # null x
    rc = L.lib.moe_hier_forward(ctypes.byref(d), fake, fake, None, fake, gm.ctypes.data, fake, fake,
                                fake, None, fake, None, None, None, None, fake, 1 << 30, None)
    assert rc == L.MOE_ERR_INVALID                                     # rank 4 but no residual
    assert L.status_string(L.MOE_ERR_TIMEOUT) == "device-side wait timed out"


def test_product_path_does_not_import_oracle():
    code = ("import sys; sys.path.insert(0, %r); import compressed_expert_two_b300.layer, "
            "compressed_expert_two_b300._lib; import bench; "
            "assert not any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules), "
            "sorted(m for m in sys.modules if m.startswith('oracle'))" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_test_aids_validate_on_the_host(L):
    assert L.lib.moe_hier_debug_set_wait(0, -1) == L.MOE_ERR_INVALID
    import numpy as np
    d = desc_for(L)                                  # an FP32 layer: no tensor-core router
    gm = np.array([0, 0, 0, 0, 1, 1, 1, 1], dtype=np.int32)
    fake = 1 << 20
    rc = L.lib.moe_hier_debug_route_tc(ctypes.byref(d), fake, fake, None, fake, gm.ctypes.data, fake, fake,
                                       1 << 30, None)
    assert rc == L.MOE_ERR_UNSUPPORTED


def test_binding_arity_matches_header(L):
    """Every ctypes binding declares as many arguments as the header's prototype (a missing one
    shifts the stream handle and crashes the host)."""
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "moehier.h")).read(), flags=re.S)
    protos = re.findall(r"\b(?:int|size_t|const char\*)\s+(moe_hier_\w+)\s*\(([^;]*?)\);", src, flags=re.S)
    assert len(protos) >= 14
    for name, params in protos:
        params = params.strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        assert len(getattr(L.lib, name).argtypes) == n, name
