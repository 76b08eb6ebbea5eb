"""Idle-group offload (moe_hier_offload_*): group bases in pinned host memory, a device cache of
fewer slots than groups, groups copied in when a batch hits them ("Breaking the MoE LLM
Trilemma", paper notes, key design 4: idle groups off the GPU, brought back when used).

Bars: every batch's output equals, bit for bit, the resident-weight forward pass on the same x
(same kernels; only the base addresses differ), and one batch matches the oracle within the layer
tolerance; the cache contents, copies and hits follow an independent re-statement of the
replacement rule (empty slot first, else the least recently used slot whose group the batch does
not hit); the batches run both one after another and pipelined (batch i+1 routed, and its
missing groups copied, while batch i's FFN runs, two workspaces).
"""
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


def layer_cfg(T):
    return MoEConfig("offload", T=T, d=512, f=1024, E=32, G=8, kg=1, ke=2, r=16, dtype="bf16", resid="int4",
                     group_map="contiguous", seed=71, zipf_s=1.2, resid_std=0.2)


class LRU:
    """The replacement rule, restated: hit groups already cached are touched; each missing hit group
    takes an empty slot (lowest index), else the least recently touched slot whose group is not hit."""

    def __init__(self, slots):
        self.slot_group = [-1] * slots
        self.last = [0] * slots
        self.tick = 0
        self.misses = self.hits = 0

    def require(self, hit):
        self.tick += 1
        need = [g for g in range(len(hit)) if hit[g]]
        for g in need:
            if g in self.slot_group:
                self.last[self.slot_group.index(g)] = self.tick
                self.hits += 1
        for g in need:
            if g in self.slot_group:
                continue
            empty = [s for s, og in enumerate(self.slot_group) if og < 0]
            if empty:
                v = empty[0]
            else:
                cand = [s for s, og in enumerate(self.slot_group) if og not in need]
                v = min(cand, key=lambda s: self.last[s])
            self.slot_group[v] = g
            self.last[v] = self.tick
            self.misses += 1


def setup(L, T, slots):
    from compressed_expert_two_b300.layer import DeviceLayer
    cfg = layer_cfg(T)
    inp = make_inputs(cfg)
    layer = DeviceLayer(inp, device="cuda")
    host = {m: inp["w_" + m].contiguous().pin_memory() for m in ("gate", "up", "down")}
    cache = {m: torch.empty((slots,) + tuple(inp["w_" + m].shape[1:]), dtype=torch.bfloat16, device="cuda")
             for m in ("gate", "up", "down")}
    off = L.Offload(layer.desc, host["gate"], host["up"], host["down"], cache["gate"], cache["up"], cache["down"],
                    slots)
    return cfg, inp, layer, off, host, cache


def batches(cfg, n, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(cfg.T, cfg.d, generator=g).to(torch.bfloat16).cuda() for _ in range(n)]


def offload_step(L, layer, off, x, ws, copy_stream, stream):
    """route, permute, hit groups, copies, FFN from the cache, combine: returns (y, hit, copied).
    The batch's device buffers stay referenced from y (keep_alive) until the caller drops y, so
    that no later allocation reuses them while a stream may still read them."""
    cfg = layer.cfg
    o = layer.new_outputs()
    L.moe_hier_route(layer.desc, x, layer.w_group, layer.b_group, layer.w_expert, layer.group_map, o["gidx"],
                     o["eidx"], o["gate"], ws, layer.ws_bytes, stream)
    p = {k: torch.empty(n, dtype=torch.int32, device="cuda") for k, n in
         (("row_asg", cfg.T * cfg.kg), ("row_begin", cfg.G + 1))}
    L.moe_hier_permute(layer.desc, layer.group_map, o["eidx"], None, None, None, None, None, p["row_asg"], None,
                       p["row_begin"], ws, layer.ws_bytes, stream)
    hit = off.groups_hit(p["row_begin"], stream)
    copied = off.require(hit, copy_stream)
    y = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    off.ffn(layer.desc, x, layer.group_map, layer.resid, o["eidx"], o["gate"], p["row_asg"], p["row_begin"], y, ws,
            layer.ws_bytes, stream)
    KEEP.append((o, p))
    return y, hit, copied


KEEP = []


def test_offload_batches_match_resident_forward_and_the_replacement_rule(L):
    cfg, inp, layer, off, host, cache = setup(L, T=3, slots=3)
    copy = torch.cuda.Stream()
    stream = torch.cuda.current_stream().cuda_stream
    lru = LRU(3)
    try:
        for i, x in enumerate(batches(cfg, 12, seed=5)):
            y, hit, copied = offload_step(L, layer, off, x, layer.ws, copy.cuda_stream, stream)
            want = layer.forward(x=x)["y"]
            torch.cuda.synchronize()
            assert torch.equal(y, want), i
            before = lru.misses
            lru.require(hit)
            st = off.stats()
            assert copied == lru.misses - before
            assert st["slot_group"] == lru.slot_group and st["misses"] == lru.misses and st["hits"] == lru.hits
            assert st["bytes_copied"] == lru.misses * 3 * cfg.d * cfg.f * 2
            if i == 0:      # one batch against the oracle, too
                sub = dict(inp)
                sub["x"] = x.cpu()
                ref = oracle.forward(sub)
                yr = ref["y"]
                err = np.abs(y.float().cpu().numpy() - yr)
                assert err.max() <= 2e-2 * np.abs(yr).max() and err.sum() <= 5e-3 * np.abs(yr).sum()
        assert lru.hits > 0 and lru.misses > 3          # the sequence both reuses and evicts
    finally:
        off.close()


def test_offload_pipelined_batches(L):
    """Batch i+1 is routed and its missing groups copied while batch i's FFN may still run (two
    workspaces, two compute streams): every output still equals the resident forward pass."""
    cfg, inp, layer, off, host, cache = setup(L, T=3, slots=3)
    copy = torch.cuda.Stream()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [layer.ws, torch.zeros_like(layer.ws)]
    xs = batches(cfg, 10, seed=6)
    ys = []
    try:
        for i, x in enumerate(xs):
            s = streams[i & 1]
            s.wait_stream(torch.cuda.current_stream())
            y, _, _ = offload_step(L, layer, off, x, wss[i & 1], copy.cuda_stream, s.cuda_stream)
            ys.append(y)
        torch.cuda.synchronize()
        for i, x in enumerate(xs):
            assert torch.equal(ys[i], layer.forward(x=x)["y"]), i
        torch.cuda.synchronize()
    finally:
        off.close()


def test_offload_rejects_more_hit_groups_than_slots(L):
    cfg, inp, layer, off, host, cache = setup(L, T=3, slots=3)
    try:
        with pytest.raises(L.MoeError):
            off.require(np.ones(cfg.G, dtype=np.int32), torch.cuda.current_stream().cuda_stream)
    finally:
        off.close()
