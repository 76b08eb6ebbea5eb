"""Device-resident layer: uploads a layer's tensors once and calls the C ABI on torch's stream.

PyTorch supplies device memory and the stream; every step of the layer runs in libmoehier.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib as L


def make_desc(cfg, T: Optional[int] = None) -> L.MoeHierDesc:
    return L.MoeHierDesc(T=cfg.T if T is None else T, d_model=cfg.d, d_ff=cfg.f, E=cfg.E, G=cfg.G,
                         topk_group=cfg.kg, topk_expert=cfg.ke, rank=cfg.r,
                         act_dtype=L.MOE_BF16 if cfg.dtype == "bf16" else L.MOE_F32,
                         resid_fmt=L.MOE_RESID_INT4_G64 if cfg.resid == "int4" else L.MOE_RESID_F32,
                         route_mode=L.MOE_ROUTE_ACROSS if getattr(cfg, "route", "within") == "across"
                         else L.MOE_ROUTE_WITHIN)


class DeviceLayer:
    """Holds the weights of one layer on ``device`` plus a workspace sized for ``T`` tokens."""

    def __init__(self, inp: dict, device="cuda", T: Optional[int] = None):
        cfg = inp["cfg"]
        self.cfg = cfg
        self.device = torch.device(device)
        dev = self.device
        self.T = cfg.T if T is None else T
        self.desc = make_desc(cfg, self.T)
        self.x = inp["x"].to(dev).contiguous() if inp["x"].shape[0] == self.T else None
        self.w_group = inp["w_group"].to(dev).contiguous()
        self.b_group = inp["b_group"].to(dev).contiguous() if inp["b_group"] is not None else None
        self.w_expert = inp["w_expert"].to(dev).contiguous()
        self.group_map = inp["group_map"].to(torch.int32).contiguous()      # host
        self.w_gate = inp["w_gate"].to(dev).contiguous()
        self.w_up = inp["w_up"].to(dev).contiguous()
        self.w_down = inp["w_down"].to(dev).contiguous()
        self._resid_t = {}
        self.resid = L.MoeHierResid()
        for m_i, m in enumerate(("gate", "up", "down")):
            rm = inp["resid"][m]
            if cfg.resid == "int4":
                t = {k: v.to(dev).contiguous() for k, v in rm.items()}
                self.resid.A[m_i], self.resid.B[m_i] = t["Aq"].data_ptr(), t["Bq"].data_ptr()
                self.resid.sA[m_i], self.resid.sB[m_i] = t["As"].data_ptr(), t["Bs"].data_ptr()
            else:
                t = {k: v.to(dev).contiguous() for k, v in rm.items()}
                self.resid.A[m_i], self.resid.B[m_i] = t["A"].data_ptr(), t["B"].data_ptr()
            self._resid_t[m] = t
        self.ws_bytes = L.moe_hier_workspace_size(self.desc)
        self.ws = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.act_dtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32

    @property
    def stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def new_outputs(self):
        cfg, T, dev = self.cfg, self.T, self.device
        return {"y": torch.empty(T, cfg.d, dtype=self.act_dtype, device=dev),
                "gidx": torch.empty(T, cfg.kg, dtype=torch.int32, device=dev),
                "eidx": torch.empty(T, cfg.k, dtype=torch.int32, device=dev),
                "gate": torch.empty(T, cfg.k, dtype=torch.float32, device=dev),
                "perm": torch.empty(T * cfg.k, dtype=torch.int32, device=dev)}

    def forward(self, x=None, out=None, routing_out: bool = True):
        x = self.x if x is None else x
        o = self.new_outputs() if out is None else out
        L.moe_hier_forward(self.desc, x, self.w_group, self.b_group, self.w_expert, self.group_map,
                           self.w_gate, self.w_up, self.w_down, self.resid, o["y"],
                           o["gidx"] if routing_out else None, o["eidx"] if routing_out else None,
                           o["gate"] if routing_out else None, o["perm"] if routing_out else None,
                           self.ws, self.ws_bytes, self.stream)
        return o

    def prepare(self):
        """Builds the residual stacks once (moe_hier_prepare); forward(prepared=True) then reads them."""
        self.prep_bytes = L.moe_hier_prepared_size(self.desc)
        self.prep = torch.empty(max(self.prep_bytes, 256), dtype=torch.uint8, device=self.device)
        L.moe_hier_prepare(self.desc, self.group_map, self.resid, self.prep, self.prep_bytes, self.stream)
        return self

    def forward_prepared(self, x=None, out=None, routing_out: bool = True):
        x = self.x if x is None else x
        o = self.new_outputs() if out is None else out
        L.moe_hier_forward_prepared(self.desc, x, self.w_group, self.b_group, self.w_expert, self.group_map,
                                    self.w_gate, self.w_up, self.w_down, self.resid, self.prep, self.prep_bytes,
                                    o["y"], o["gidx"] if routing_out else None, o["eidx"] if routing_out else None,
                                    o["gate"] if routing_out else None, o["perm"] if routing_out else None,
                                    self.ws, self.ws_bytes, self.stream)
        return o

    # ---- the stages one by one (same kernels as forward) ----
    def route(self, x=None):
        x = self.x if x is None else x
        o = self.new_outputs()
        L.moe_hier_route(self.desc, x, self.w_group, self.b_group, self.w_expert, self.group_map,
                         o["gidx"], o["eidx"], o["gate"], self.ws, self.ws_bytes, self.stream)
        return o

    def permute(self, eidx):
        cfg, T, dev = self.cfg, self.T, self.device
        i32 = dict(dtype=torch.int32, device=dev)
        p = {"perm": torch.empty(T * cfg.k, **i32), "inv_pos": torch.empty(T * cfg.k, **i32),
             "expert_begin": torch.empty(cfg.E, **i32), "expert_count": torch.empty(cfg.E, **i32),
             "group_begin": torch.empty(cfg.G + 1, **i32), "row_asg": torch.empty(T * cfg.kg, **i32),
             "row_of": torch.empty(T * cfg.kg, **i32), "row_begin": torch.empty(cfg.G + 1, **i32)}
        L.moe_hier_permute(self.desc, self.group_map, eidx, p["perm"], p["inv_pos"], p["expert_begin"],
                           p["expert_count"], p["group_begin"], p["row_asg"], p["row_of"],
                           p["row_begin"], self.ws, self.ws_bytes, self.stream)
        return p

    def ffn(self, x, eidx, gate, row_asg, row_begin):
        cfg, T = self.cfg, self.T
        y_rows = torch.empty(T, cfg.kg, cfg.d, dtype=self.act_dtype, device=self.device)
        L.moe_hier_ffn(self.desc, x, self.group_map, self.w_gate, self.w_up, self.w_down, self.resid,
                       eidx, gate, row_asg, row_begin, y_rows, self.ws, self.ws_bytes, self.stream)
        return y_rows

    def combine(self, y_rows):
        y = torch.empty(self.T, self.cfg.d, dtype=self.act_dtype, device=self.device)
        L.moe_hier_combine(self.desc, y_rows, y, self.stream)
        return y

    def status(self) -> int:
        return L.moe_hier_get_status(self.ws, self.stream)
