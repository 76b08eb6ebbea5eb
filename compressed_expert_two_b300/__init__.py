"""Clustered, compressed MoE layer forward pass for NVIDIA B300 (sm_103a).

The layer runs in libmoehier.so (hand-written CUDA behind a C ABI, declared in include/moehier.h).
``compressed_expert_two_b300._lib`` binds the C entry points under their own names and
``compressed_expert_two_b300.layer.DeviceLayer`` keeps a layer's tensors on the device.  Both
raise ImportError when the library has not been built (``python -m compressed_expert_two_b300.build``).
"""


def __getattr__(name):
    if name in ("DeviceLayer", "make_desc"):
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
