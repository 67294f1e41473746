"""CPU oracle for NVFP4 / MXFP4 block-scaled quantisation and GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only
the test-suite, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code, header, table or constant generator with the CUDA path.

It is plain numpy: fp32 where the method fixes fp32 arithmetic (the quantiser,
one IEEE-rounded operation at a time, no fused multiply-add), fp64 for the GEMM.
Each function cites the passage it follows as "page title, section".  Sources:

* [vLLM-SM103] vLLM fork compare view "add pdl" (sm103 branch): the quant
  kernel (nvfp4_quant_kernels.cu, "SM103 (B300) activation quantization
  kernel"), the scale-layout conversion kernels ("Scale factor layout
  conversion: SM100 <-> SM103"), the GEMM entry ("SM103 Entry Point"), the
  SM103 layout helper (nvfp4_utils.cuh) and the quant test
  (test_nvfp4_quant.py, "SM103-native quantization correctness").
* [FI-4865] FlashInfer PR 4865 "perf(gemm): optimize SM103 CuTe DSL mm_fp4
  kernel", section "2. Alpha epilogue bug".
* [FI-4466] FlashInfer PR 4466 "sm100 cute_dsl w4a16 gemm", follow-up PR 4620
  text (the 6-D strided scale view over the 128x4-swizzled buffer).
* [vLLM-51158] vLLM PR 51158 "Enable CUTLASS MXFP4 W4A4 MoE on SM12x".

Readings taken where the pages are silent:
quantiser operation order, sign of zero for e2m1, nibble order, e4m3
saturation and the MXFP4 scale rounding (round up to a power of two).
Parity pins: every function here is pinned by tests/test_oracle_*.py.
"""
from . import formats, layout, quant, gemm, moe  # noqa: F401
