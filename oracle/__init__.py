"""CPU oracle for the FP8 lightning indexer: test infrastructure, not product code.

This package is a plain, slow, deliberately unoptimised restatement of what the
indexer computes, written from the source pages' statement of the method:

* "DeepSeek V3.2 稀疏注意力 DSA 推理流程图解" (aiinfra.pub): the cost table,
  the data-flow section, and "Indexer 内部到底做了什么" (the six steps inside
  the indexer, in particular step ⑤ fused k quantisation + cache insert and
  step ⑥ the logit definition and top-2048 selection).
* "V4.1 索引器接入稀疏 MQA logits" (prhub.com.cn review of vLLM PR #56254):
  the 实现拆解 (implementation) section and the 关键源码片段 (key source
  snippets) section for candidate expansion, the sparse top-k and the remap.
* "修复 DSV4 FlashInfer 稀疏 MLA 在打包 KV 布局下的地址错误" (prhub.com.cn
  review of vLLM PR #47493): the 实现拆解 section and the remap snippet for
  block-span slot conversion.

Floating point is evaluated in fp64 unless the method fixes a narrower precision
(the fp32 quantisation scale, the e4m3 and bf16 encodings).

Only the test suite, the smoke entry point and the benchmark's CPU-baseline leg
may import this package. The GPU library shares no code with it.

Every function here is pinned by a test under ``tests/`` against something other
than itself (format definitions, closed forms, brute force, library routines on
special cases). No function is "parity unpinned".
"""

from . import codecs, indexer  # noqa: F401
