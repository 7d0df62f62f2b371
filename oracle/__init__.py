"""fp64 CPU oracle for the attention forward pass.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import anything under
``oracle/``. The product (the CUDA library and its Python binding) never
does, and shares no code with it.

Contents:
  attn        -- ctypes loader of the C reference (exact definition, fp64).
  tiled_model -- fp64 model of the tile-by-tile online softmax with the
                 conditional (lazy) rescale, in the pages' order.
  exp2_emu    -- model of the software 2^x (Cody-Waite range reduction +
                 Horner polynomial) with its own minimax fit.
  splitkv     -- fp64 key-range forward and the LSE-weighted combine.
  attn_bwd    -- fp64 gradient of attention (dQ, dK, dV) by the definition.
  fp8         -- e4m3 decoding and the fp64 forward of dequantised FP8
                 inputs, with the error bound of rounding P to e4m3.
"""
