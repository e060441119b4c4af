"""CPU oracle for the routed-expert MoE decode path and its NVFP4 prompt-path GEMM.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, numpy restatement of
what the method computes, written from the pages that describe it:

  * FreeToken PR #704, "serve GGUF experts on the cpu and hybrid backends
    through ggml-cpu" -- section "How it plugs into the CPU executor" (the
    prep_input -> gate_up -> prep_inter -> down pipeline and the route sum);
  * FreeToken PR #732, "apply the weight scales of nvfp4 gguf tensors" --
    section "Design" (the per-expert [E,4] scale bank and the layer formula);
  * Strata PR #292, "NVFP4 routed experts: converter, pack, decode, prompt path
    (W4A8, W4A4 on Blackwell), AVX-512 CPU rows" -- section "Summary/Pipeline"
    (q8_1 activations, software UE4M3/E2M1 decode, each global scale applied to
    its own projection's fp32 output, W4A8/W4A4 prompt modes);
  * FreeToken issue #194, "avoid max-stride padding for heterogeneous GGUF
    expert banks" -- section "Reproduction geometry" (Q4_K/BF16 row sizes).

Arithmetic is fp64 except where a step is defined in a narrower type (the
fp32 q8_1 quantizer, fp16 block scales, the final bf16 output).  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it; the product library never calls into it and shares no code with it.

Parity status per function is stated in each module header.
"""
