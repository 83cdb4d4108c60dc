"""CPU oracle for scaled-FP8 matrix multiply -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement of what the
scaled-FP8 path computes, in numpy with float64 (float32 where the method
itself fixes fp32 arithmetic, e.g. ``x / scale`` in the quantizer).  It exists
to check the CUDA library and is never part of the product path: only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
legs import it.  It shares no code with the CUDA path (no kernels, headers,
helpers or constant tables); both sides only share the seeded input generators
in ``workloads.py``.

Sources (web pages, cited by title and section):

* "Flax FP8 量化实战指南" (Flax FP8 guide, 0539edu.com/news/4761306):
  section 1 (Q/DQ), 2.2 (current scaling, ``quantize``/``dequantize``),
  2.3 (delayed scaling, ``compute_amax_history``/``update_fp8_meta``),
  5.1 (meta state), 5.3 (the ``fp32_max_grad`` worked example).
* "Nanochat的FP8训练模块" (nanochat FP8 module, lzwjava.github.io), section
  "实现": forward/backward GEMMs, E5M2 gradients with max 57344, TN layout.
* "Transformers 中的细粒度 FP8 量化配置..." (Transformers fine-grained FP8,
  m.nxbn.cn/news/32317): section 一 (128x128 weight blocks, 1x128 activation
  groups), section 七 (UE8M0 scales rounded up, quantize with the rounded scale).
* "MOSS: 高效、精确的 FP8 LLM 训练" (MOSS blog, blog.daoxuan.cc/posts/50279):
  section 2 (SNR), section 4 (two-level microscaling).

Modules: ``formats`` (E4M3fn / E5M2 / E8M0 codecs), ``quantize`` (the four
quantization granularities), ``delayed`` (amax-history state machine),
``gemm`` (float64 dequantized GEMM and its error bound), ``snr``,
``training`` (SwiGLU MLP and AdamW, support arithmetic for the training
workload).  Parity status of each function is stated in its module header.
"""
