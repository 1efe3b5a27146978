"""CPU oracle for the routed-MoE layer.  TEST INFRASTRUCTURE ONLY.

This package is the slow, plain reference that the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library never does, and it shares no
code with the library (the seeded input generator in ``synth`` feeds both).

It computes the layer literally, following the colibrì pages:

* router  -- "Colibri (colibrì): GLM-5.2 local inference on 25 GB of RAM",
  section "How it works (validated core mechanics)": sigmoid affinities, a
  correction bias used for ranking only, lower expert id wins a tie, gate
  weights renormalised from the unbiased sigmoid, non-finite input rejected;
  plus the group-limited top-k of the DeepSeek-V3 ``noaux_tc`` pattern that
  the same page and the colibrì v1.0 README ("What's implemented") name.
* Q8_0-style activations, packed int4 / packed int2 / int8 per-row-scaled
  weights, the SwiGLU expert and the batch-union evaluation -- colibrì v1.0 README,
  "What's implemented" (integer-dot kernels, quantization kernels,
  batch-union MoE) and "Experimental Metal backend" (routed-expert SwiGLU).
* the routing-weighted combine plus the always-on shared expert -- the
  router description on the GLM-5.2 write-up ("Colibri (colibrì): GLM-5.2 local inference on 25 GB of RAM") and "What's implemented".

Floating point is fp64 except where a floating-point value decides an
integer code (the Q8_0 scale and rounding), which is done in fp32 exactly as
the kernel does it.  Integer block dot products are exact (fp64 products of
8-bit codes are exact integers; returned as int64).

Readings of points the pages leave open are listed in the docstrings of the
functions that take them.  Parity status: every function here is pinned by
the tests under ``tests/test_oracle_*.py`` (closed forms, hand-worked
examples, brute force, invariants); the final fp32 layer outputs have no
printed worked example on the pages and are pinned only through those
invariants and the fp64 dequantised bound.
"""
from .quant import (q8_0_quantize, q8_0_dequantize, q8_0_stable_mask,
                    int4_pack, int4_unpack, int2_pack, int2_unpack,
                    unpack_weight_rows)
from .router import (router_logits, route, route_margins, sigmoid)
from .expert import block_dots, expert_ffn, expert_ffn_dequant_fp64
from .layer import (union_tables, moe_forward, moe_layer, dense_reference)

__all__ = [
    "q8_0_quantize", "q8_0_dequantize", "q8_0_stable_mask", "int4_pack",
    "int4_unpack", "int2_pack", "int2_unpack", "unpack_weight_rows", "router_logits", "route",
    "route_margins", "sigmoid", "block_dots", "expert_ffn",
    "expert_ffn_dequant_fp64", "union_tables", "moe_forward", "moe_layer",
    "dense_reference",
]
