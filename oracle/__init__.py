"""CPU oracle for KIVI-style KV-cache quantization and decode attention.

TEST INFRASTRUCTURE.  This package is the slow, plain reference that the CUDA
library is checked against.  Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference leg may import it; the library itself
never does, and it shares no code, tables or helpers with the CUDA sources.

Sources (the three web pages this method is taken from):
  [explainer]  KIVI explainer, discosf.com/news/3594501 (page titled
               "企业官网建设流程全解析"), sections 2.1, 2.2, 3.1, 3.2, 5.2.
  [axis-guide] "KV cache quantization axis selection guide", unite.ai (zh-cn),
               sections "量化错误的真正组成" (what quantization error is made
               of), "键：异常值位于固定通道中" (keys: outliers sit in fixed
               channels), "值：直觉在哪里破裂" (values: where intuition breaks),
               "系统税收" (the system tax).
  [survey]     "3.2.3 KV Cache Quantization", blog.csdn.net (KIVI: keys per
               channel, values per token, 2 bits, no fine-tuning).

Modules:
  quant      uniform asymmetric B-bit group quantizer; key / value grouping
  cache      streaming cache state: prefill split, fp16 residual, flush
  attention  fp64 single-query decode attention over the dequantized cache
  layout     packing of codes / scales / zeros into the library's byte layout
  accounting closed-form byte counts

Parity status of each function is stated in its module docstring.
"""
