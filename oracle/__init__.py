"""CPU oracle for the clustered, compressed MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product path (the C-ABI library and its Python binding) never imports, calls or
links anything here, and this package imports nothing from the product path; the two share only
the seeded input generator in ``synth``.

Parity status per function (pins live in ``tests/test_oracle_pins.py``):
  canonical_logits  -- pinned (exact small-integer sums, hand-derived rounding cases, FP64 bound)
  route             -- pinned (brute force over every routing choice, gate sum, k=1 gate == 1,
                       torch.topk/softmax special case for G == 1)
  permute           -- pinned (invariants, brute-force sorted(), inverse bijection)
  dequant_int4      -- pinned (nibble convention worked by hand from the INT4 unpack listing)
  forward / forward_tokens -- pinned (factor identity, r = 0 dense group-base MoE against a torch
                       FP64 SwiGLU, K = 1 / r = 0 textbook top-k MoE, brute-force output check)
  compress.group_mean_base / tsvd / quantise_int4_g64 / reconstruction_error / compress_matrix
                    -- pinned (tests/test_compress_oracle.py): exact integer means and a
                       hand-derived FP32 order case, a constructed spectrum and a diagonal matrix
                       for the truncated SVD, the input generator's independent packer and the
                       golden INT4 byte for the quantiser, K = 1 reconstructs exactly
  compression_ratio -- pinned to the closed form at d=4096, K=8, r=16 (7.53x); the page's printed
                       "about 6.6x" disagrees with its own formula: that figure is parity unpinned.
"""
from . import compress
from .moe import (canonical_logits, route, permute, dequant_int4, resid_dense, materialise,
                  forward, forward_tokens, compression_ratio, param_counts, silu)

__all__ = ["compress", "canonical_logits", "route", "permute", "dequant_int4", "resid_dense", "materialise",
           "forward", "forward_tokens", "compression_ratio", "param_counts", "silu"]
