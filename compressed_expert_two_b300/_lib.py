"""ctypes binding of libmoehier.so: the C-ABI entry points under the same names.

Argument marshalling only (tensor -> device pointer, dataclass -> C struct).  Every step of the
layer runs in the library's CUDA kernels; there is no fallback.  Importing this module fails
loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoehier.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = \
    0, -1, -2, -3, -4, -5
MOE_F32, MOE_BF16 = 0, 1
MOE_RESID_F32, MOE_RESID_INT4_G64 = 0, 1
MOE_ROUTE_WITHIN, MOE_ROUTE_ACROSS = 0, 1


class MoeHierDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("G", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("topk_expert", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("resid_fmt", ctypes.c_int32),
                ("route_mode", ctypes.c_int32)]


class MoeHierCompressDesc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("G", ctypes.c_int32), ("d_out", ctypes.c_int32),
                ("d_in", ctypes.c_int32), ("rank", ctypes.c_int32), ("sketch", ctypes.c_int32),
                ("power_iters", ctypes.c_int32)]


class MoeHierResid(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p * 3), ("B", ctypes.c_void_p * 3),
                ("sA", ctypes.c_void_p * 3), ("sB", ctypes.c_void_p * 3)]


EXPORTS = ["moe_hier_workspace_size", "moe_hier_route", "moe_hier_permute", "moe_hier_ffn",
           "moe_hier_combine", "moe_hier_forward", "moe_hier_get_status", "moe_hier_status_string",
           "moe_hier_last_cuda_error", "moe_hier_profile_begin", "moe_hier_profile_end",
           "moe_hier_debug_set_wait", "moe_hier_debug_route_tc", "moe_hier_permute_noalloc",
           "moe_hier_compress_workspace_size", "moe_hier_compress", "moe_hier_quantise_int4",
           "moe_hier_offload_create", "moe_hier_offload_destroy", "moe_hier_groups_hit",
           "moe_hier_offload_require", "moe_hier_ffn_offload", "moe_hier_offload_stats",
           "moe_hier_prepared_size", "moe_hier_prepare", "moe_hier_forward_prepared"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        detail = status_string(code)
        if code == MOE_ERR_CUDA:
            detail += ": " + lib.moe_hier_last_cuda_error().decode()
        super().__init__(f"{fn} failed: {code} ({detail})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoehier.so is not built ({LIB_PATH}); run "
                          "`python -m compressed_expert_two_b300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D, Rp = ctypes.POINTER(MoeHierDesc), ctypes.POINTER(MoeHierResid)
    lib.moe_hier_workspace_size.argtypes = [D, ctypes.POINTER(ctypes.c_int)]
    lib.moe_hier_workspace_size.restype = S
    lib.moe_hier_route.argtypes = [D, P, P, P, P, P, P, P, P, P, S, P]
    lib.moe_hier_permute.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, S, P]
    lib.moe_hier_ffn.argtypes = [D, P, P, P, P, P, Rp, P, P, P, P, P, P, S, P]
    lib.moe_hier_combine.argtypes = [D, P, P, P]
    lib.moe_hier_forward.argtypes = [D, P, P, P, P, P, P, P, P, Rp, P, P, P, P, P, P, S, P]
    lib.moe_hier_get_status.argtypes = [P, P]
    lib.moe_hier_profile_begin.argtypes = [ctypes.POINTER(ctypes.c_void_p), I]
    lib.moe_hier_profile_end.argtypes = [ctypes.POINTER(ctypes.c_char_p), I]
    lib.moe_hier_status_string.argtypes = [I]
    lib.moe_hier_status_string.restype = ctypes.c_char_p
    C = ctypes.POINTER(MoeHierCompressDesc)
    lib.moe_hier_compress_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_int)]
    lib.moe_hier_compress_workspace_size.restype = S
    lib.moe_hier_compress.argtypes = [C] + [P] * 13 + [S, P]
    lib.moe_hier_quantise_int4.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, P, P]
    lib.moe_hier_prepared_size.argtypes = [D, ctypes.POINTER(ctypes.c_int)]
    lib.moe_hier_prepared_size.restype = S
    lib.moe_hier_prepare.argtypes = [D, P, Rp, P, S, P]
    lib.moe_hier_forward_prepared.argtypes = [D, P, P, P, P, P, P, P, P, Rp, P, S, P, P, P, P, P, P, S, P]
    lib.moe_hier_offload_create.argtypes = [D, P, P, P, P, P, P, ctypes.c_int32, ctypes.POINTER(P)]
    lib.moe_hier_offload_destroy.argtypes = [P]
    lib.moe_hier_groups_hit.argtypes = [D, P, P, P]
    lib.moe_hier_offload_require.argtypes = [P, P, P, P]
    lib.moe_hier_ffn_offload.argtypes = [P, D, P, P, Rp, P, P, P, P, P, P, S, P]
    U64p = ctypes.POINTER(ctypes.c_uint64)
    lib.moe_hier_offload_stats.argtypes = [P, U64p, U64p, U64p, P]
    lib.moe_hier_debug_set_wait.argtypes = [ctypes.c_uint64, I]
    lib.moe_hier_debug_route_tc.argtypes = [D, P, P, P, P, P, P, P, S, P]
    lib.moe_hier_permute_noalloc.argtypes = [D] + [P] * 11
    lib.moe_hier_last_cuda_error.argtypes = []
    lib.moe_hier_last_cuda_error.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("moe_hier_workspace_size", "moe_hier_status_string", "moe_hier_last_cuda_error",
                        "moe_hier_compress_workspace_size", "moe_hier_prepared_size"):
            getattr(lib, name).restype = I
    return lib


lib = _load()


def _p(t) -> Optional[int]:
    """Device (or host) address of a tensor; None for None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def status_string(code: int) -> str:
    return lib.moe_hier_status_string(code).decode()


def moe_hier_workspace_size(desc: MoeHierDesc) -> int:
    st = ctypes.c_int(0)
    n = lib.moe_hier_workspace_size(ctypes.byref(desc), ctypes.byref(st))
    _check("moe_hier_workspace_size", st.value)
    return n


def moe_hier_route(desc, x, w_group, b_group, w_expert, group_map_host, gidx, eidx, gate, ws, ws_bytes, stream):
    _check("moe_hier_route", lib.moe_hier_route(
        ctypes.byref(desc), _p(x), _p(w_group), _p(b_group), _p(w_expert), _p(group_map_host),
        _p(gidx), _p(eidx), _p(gate), _p(ws), ws_bytes, stream))


def moe_hier_permute(desc, group_map_host, eidx, perm, inv_pos, expert_begin, expert_count,
                     group_begin, row_asg, row_of, row_begin, ws, ws_bytes, stream):
    _check("moe_hier_permute", lib.moe_hier_permute(
        ctypes.byref(desc), _p(group_map_host), _p(eidx), _p(perm), _p(inv_pos), _p(expert_begin),
        _p(expert_count), _p(group_begin), _p(row_asg), _p(row_of), _p(row_begin), _p(ws),
        ws_bytes, stream))


def moe_hier_ffn(desc, x, group_map_host, w_gate, w_up, w_down, resid, eidx, gate, row_asg,
                 row_begin, y_rows, ws, ws_bytes, stream):
    _check("moe_hier_ffn", lib.moe_hier_ffn(
        ctypes.byref(desc), _p(x), _p(group_map_host), _p(w_gate), _p(w_up), _p(w_down),
        ctypes.byref(resid), _p(eidx), _p(gate), _p(row_asg), _p(row_begin), _p(y_rows), _p(ws),
        ws_bytes, stream))


def moe_hier_combine(desc, y_rows, y, stream):
    _check("moe_hier_combine", lib.moe_hier_combine(ctypes.byref(desc), _p(y_rows), _p(y), stream))


def moe_hier_forward(desc, x, w_group, b_group, w_expert, group_map_host, w_gate, w_up, w_down,
                     resid, y, gidx, eidx, gate, perm, ws, ws_bytes, stream):
    _check("moe_hier_forward", lib.moe_hier_forward(
        ctypes.byref(desc), _p(x), _p(w_group), _p(b_group), _p(w_expert), _p(group_map_host),
        _p(w_gate), _p(w_up), _p(w_down), ctypes.byref(resid), _p(y), _p(gidx), _p(eidx),
        _p(gate), _p(perm), _p(ws), ws_bytes, stream))


def moe_hier_prepared_size(desc: MoeHierDesc) -> int:
    st = ctypes.c_int(0)
    n = lib.moe_hier_prepared_size(ctypes.byref(desc), ctypes.byref(st))
    _check("moe_hier_prepared_size", st.value)
    return n


def moe_hier_prepare(desc, group_map_host, resid, prep, prep_bytes, stream):
    _check("moe_hier_prepare", lib.moe_hier_prepare(ctypes.byref(desc), _p(group_map_host), ctypes.byref(resid),
                                                    _p(prep), prep_bytes, stream))


def moe_hier_forward_prepared(desc, x, w_group, b_group, w_expert, group_map_host, w_gate, w_up, w_down, resid,
                              prep, prep_bytes, y, gidx, eidx, gate, perm, ws, ws_bytes, stream):
    _check("moe_hier_forward_prepared", lib.moe_hier_forward_prepared(
        ctypes.byref(desc), _p(x), _p(w_group), _p(b_group), _p(w_expert), _p(group_map_host), _p(w_gate),
        _p(w_up), _p(w_down), ctypes.byref(resid), _p(prep), prep_bytes, _p(y), _p(gidx), _p(eidx), _p(gate),
        _p(perm), _p(ws), ws_bytes, stream))


def moe_hier_profile_begin(event_handles) -> ctypes.Array:
    """Start marking kernel launches with the given cudaEvent_t handles (ints); returns the C
    array, which the caller keeps alive until moe_hier_profile_end."""
    arr = (ctypes.c_void_p * len(event_handles))(*event_handles)
    _check("moe_hier_profile_begin", lib.moe_hier_profile_begin(arr, len(event_handles)))
    return arr


def moe_hier_profile_end(max_names: int = 256) -> list:
    names = (ctypes.c_char_p * max_names)()
    n = lib.moe_hier_profile_end(names, max_names)
    return [names[i].decode() for i in range(min(n, max_names))]


def moe_hier_permute_noalloc(desc, group_map_host, eidx, perm, inv_pos, expert_begin, expert_count,
                             group_begin, row_asg, row_of, row_begin, stream):
    _check("moe_hier_permute_noalloc", lib.moe_hier_permute_noalloc(
        ctypes.byref(desc), _p(group_map_host), _p(eidx), _p(perm), _p(inv_pos), _p(expert_begin),
        _p(expert_count), _p(group_begin), _p(row_asg), _p(row_of), _p(row_begin), stream))


def moe_hier_debug_set_wait(wait_ns: int, phantom_arrivals: int) -> None:
    _check("moe_hier_debug_set_wait", lib.moe_hier_debug_set_wait(wait_ns, phantom_arrivals))


def moe_hier_debug_route_tc(desc, x, w_group, b_group, w_expert, group_map_host, out, ws, ws_bytes, stream):
    _check("moe_hier_debug_route_tc", lib.moe_hier_debug_route_tc(
        ctypes.byref(desc), _p(x), _p(w_group), _p(b_group), _p(w_expert), _p(group_map_host), _p(out),
        _p(ws), ws_bytes, stream))


def moe_hier_compress_workspace_size(desc: MoeHierCompressDesc) -> int:
    st = ctypes.c_int(0)
    n = lib.moe_hier_compress_workspace_size(ctypes.byref(desc), ctypes.byref(st))
    _check("moe_hier_compress_workspace_size", st.value)
    return n


def moe_hier_compress(desc, w, group_map_host, omega, base, A_codes, A_scales, B_codes, B_scales, sigma, err,
                      At_f32, Bt_f32, ws, ws_bytes, stream):
    _check("moe_hier_compress", lib.moe_hier_compress(
        ctypes.byref(desc), _p(w), _p(group_map_host), _p(omega), _p(base), _p(A_codes), _p(A_scales),
        _p(B_codes), _p(B_scales), _p(sigma), _p(err), _p(At_f32), _p(Bt_f32), _p(ws), ws_bytes, stream))


def moe_hier_quantise_int4(v, rows: int, n: int, codes, scales, stream):
    _check("moe_hier_quantise_int4", lib.moe_hier_quantise_int4(_p(v), rows, n, _p(codes), _p(scales), stream))


class Offload:
    """Handle of the idle-group offload manager (moe_hier_offload_*): the caller's pinned host
    bases and device cache, passed through unchanged."""

    def __init__(self, desc, w_gate_host, w_up_host, w_down_host, cache_gate, cache_up, cache_down, slots):
        self.h = ctypes.c_void_p()
        self.desc = desc
        _check("moe_hier_offload_create", lib.moe_hier_offload_create(
            ctypes.byref(desc), _p(w_gate_host), _p(w_up_host), _p(w_down_host), _p(cache_gate), _p(cache_up),
            _p(cache_down), slots, ctypes.byref(self.h)))
        self.slots = slots

    def groups_hit(self, row_begin, stream):
        import numpy as np
        hit = np.zeros(self.desc.G, dtype=np.int32)
        _check("moe_hier_groups_hit", lib.moe_hier_groups_hit(ctypes.byref(self.desc), _p(row_begin),
                                                              hit.ctypes.data, stream))
        return hit

    def require(self, hit, copy_stream) -> int:
        import numpy as np
        hit = np.ascontiguousarray(hit, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check("moe_hier_offload_require", lib.moe_hier_offload_require(self.h, hit.ctypes.data, ctypes.byref(n),
                                                                        copy_stream))
        return n.value

    def ffn(self, desc, x, group_map_host, resid, eidx, gate, row_asg, row_begin, y_rows, ws, ws_bytes, stream):
        _check("moe_hier_ffn_offload", lib.moe_hier_ffn_offload(
            self.h, ctypes.byref(desc), _p(x), _p(group_map_host), ctypes.byref(resid), _p(eidx), _p(gate),
            _p(row_asg), _p(row_begin), _p(y_rows), _p(ws), ws_bytes, stream))

    def stats(self):
        import numpy as np
        b, m, h = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
        sg = np.zeros(self.slots, dtype=np.int32)
        _check("moe_hier_offload_stats", lib.moe_hier_offload_stats(self.h, ctypes.byref(b), ctypes.byref(m),
                                                                    ctypes.byref(h), sg.ctypes.data))
        return {"bytes_copied": b.value, "misses": m.value, "hits": h.value, "slot_group": sg.tolist()}

    def close(self):
        if self.h:
            _check("moe_hier_offload_destroy", lib.moe_hier_offload_destroy(self.h))
            self.h = ctypes.c_void_p()


def moe_hier_get_status(ws, stream) -> int:
    return lib.moe_hier_get_status(_p(ws), stream)
