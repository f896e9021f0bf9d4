"""Plain, slow CPU oracle for the low-precision MoE routed-expert layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It shares no code with the CUDA library (no kernels, headers, tables or
helpers). Every function states the passage of the source pages, or the
public format specification, that it follows:

* "[BUG] Loss difference when training with FP8 vs. BF16 MoE"
  (Megatron-LM issue #1152): hybrid e4m3/e5m2 FP8, delayed scaling with an
  amax history of 1024 and the ``max`` reduction (repro steps).
* "Numerical fix for moe single grouped weight with fp8 fp4 primary weight
  and grad norm spikes" (Megatron-LM PR #5487): the MXFP8 / NVFP4 recipes,
  the grouped tensor with row-wise and column-wise data and scales, NVFP4
  packing two values per byte (coverage matrix; review comments).
* "FP8BlockQuantizer not work on TE" (TransformerEngine issue #2393): 1x128
  and 128x1 block scaling, the transpose identity, zero fill of partial
  blocks, block-aligned shapes (maintainer replies).
* "float8 moe training conversion API prototype" (pytorch/ao PR #2275):
  dynamic quantisation followed by a scaled grouped mm, SQNR checks of
  outputs and gradients against bf16 (description; testing).

Bit layouts of the number formats come from the OCP 8-bit floating point
specification (OFP8) and the OCP Microscaling (MX) v1.0 specification, which
the pages name only by recipe.

Parity pins: every function is pinned by tests under ``tests/`` (exhaustive
code enumeration, closed forms, invariants, brute force on tiny inputs).
"""
