"""CPU oracle for the fused MoE expert layer -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct definition that the GPU
path is checked against.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product (the CUDA library and its Python binding) never imports, calls or
links anything here, and this package imports nothing from the product.  The
two share only the seeded input generator in ``synth/``.

What it computes (the single-GPU fused MegaMoE expert layer):

* ``formats``  -- E4M3, E2M1 and UE8M0 decode/encode and the per-32 block
  quantiser (the recipe ``(1, 1, 32)`` of DeepGEMM ``fp8_fp4_mega_moe``,
  quoted on the digest page of sglang PR #36657, section 关键源码片段).
* ``routing``  -- per-expert counts, exclusive prefix offsets and the stable
  permutation (the counting and source-recording steps of the dispatch in
  the DeepGEMM SM90 MegaMoE dev log, Phase 2 entry).
* ``moe``      -- the layer: L1 gate/up GEMM, clamp, SwiGLU, FP8 requantisation
  of the L1 activations, L2 down GEMM, and the top-k weighted combine into a
  bf16 output, accumulated in fp64.
* ``moe_bf16`` -- the bf16 x bf16 variant of the layer (the BF16 MegaMoE kernel
  that DeepGEMM PR #451 fixes beside the FP8/FP4 one): the same steps with
  bfloat16 inputs, weights and L1 activations instead of the FP8/FP4 codes.
* ``moe_f8b``  -- the layer in the (1, 128, 128) recipe (E4M3 activations and
  weights with fp32 scales per 1 x 128 and 128 x 128 blocks; the SM90 recipe
  of the DeepGEMM SM90 MegaMoE dev log, Phase 1 entry).

Every function is pinned by CPU tests (``tests/test_oracle_*.py``) against
closed forms, library routines, brute force and exact rational arithmetic;
none is "parity unpinned".
"""
from . import formats, routing, moe, moe_bf16, moe_f8b  # noqa: F401
