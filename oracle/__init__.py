"""fp64 CPU oracle for the fused grouped expert MLP (forward + backward, BF16, MXFP8, NVFP4).

TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the benchmark's CPU
baseline leg may import this package. The product (the CUDA library and its Python binding)
never calls it, and it shares no code with the product: it is a plain, slow restatement of
what the layer computes, written from the two sources below.

Sources (cited by page title and section):
  [NV-blog]  NVIDIA technical blog "Boosting MoE Training Throughput with Advanced Fusion
             Kernels" (zh-cn: 借助高级融合内核提高 MoE 训练吞吐量): the SwiGLU equation and
             the GLU-epilogue section, the dActivation backward epilogue, device-resident
             per-group token counts, fused MXFP8 quantise/transpose.
  [TE-MoE]   "NVIDIA Transformer Engine 优化 MoE 生物基础模型训练" (Transformer Engine MoE
             article): the per-expert loop with index_add (Challenge 1), GroupedLinear
             semantics, the MXFP8 format (Challenge 2, Figure 3), ScaledSwiGLU routing-weight
             scaling and the fused GroupedLinear -> ScaledSwiGLU -> GroupedLinear op
             (Challenge 3, Figure 4).
  [MoE-summary] setupai.cc summary page "Boosting MoE Training Throughput with Advanced
             Fusion Kernels" (zh-hant): the NVIDIA hardware list (Blackwell: NVFP4).

Modules:
  oracle.mxfp8 - E4M3 encoding, E8M0 block scales, MXFP8 quantise / dequantise.
  oracle.nvfp4 - E2M1 encoding, E4M3 block scales, per-tensor scale, NVFP4 quantise /
                 dequantise, the 16-point random Hadamard rotation.
  oracle.moe   - routing, permutation maps, activations, grouped forward and backward
                 (BF16 / MXFP8 per expert; NVFP4 stage by stage, layer_nvfp4).

Every function here is pinned by a CPU test against something other than itself (closed
forms, finite differences, torch autograd in fp64, brute force, exhaustive enumeration, or
the independent per-token loop); none is "parity unpinned".
"""
