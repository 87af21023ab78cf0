"""CPU oracle for the NVFP4 quantize-and-multiply path of one linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links anything in this package.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.

The oracle is a plain, slow, obviously correct restatement of what the method
computes, written from:

* "Pretraining Large Language Models with NVFP4" (gist.science summary),
  Resumo técnico §2 Metodologia: the NVFP4 format (16-element blocks, E4M3
  block scales, an FP32 per-tensor scale), random Hadamard transforms on the
  Wgrad inputs, 2D 16x16 weight scaling, stochastic rounding of gradients with
  round-to-nearest-even elsewhere;
* the OCP Microscaling Formats specification v1.0 (E2M1 element encoding) and
  the OCP 8-bit Floating Point specification (E4M3 encoding), for the bit
  layouts the pages only name;
* Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
  (SC'11), for Philox4x32-10.

Two restatements of the same definitions, pinned by the same kinds of tests
and equal to each other bit for bit: the numpy modules below (the reference
used by most parity tests), and a plain C++17 library, ``cxx`` (source
``cxx/nvfp4_oracle.cpp``, std::thread over the host's cores, compiled with
-ffp-contract=off), which the full-size parity checks and the benchmark's CPU
baseline use.

Modules:
  cxx      ctypes binding of the C++ oracle (same function names)
  formats  E2M1 / E4M3 encode and decode, nibble packing
  philox   Philox4x32-10 counter-based generator
  rht      16x16 random Hadamard transform
  quant    tensor scale, 1x16 and 16x16 block quantization, transpose
           quantization, stochastic rounding, MMA scale-factor layout
  gemm     FP64-accumulated GEMM on dequantized operands
  linear   Fprop / Dgrad / Wgrad composition

Parity status: every function is pinned by the ``-m "not gpu"`` tests against
values the formats fix, closed forms, invariants, brute force or a library
conversion, except ``quant.swizzle_scales`` whose layout is a hardware
convention; it is pinned only through the GPU GEMM (parity unpinned on CPU).
"""

from . import formats, philox, rht, quant, gemm, linear  # noqa: F401
# oracle.cxx is imported on demand (it compiles its C++ library on first use)
