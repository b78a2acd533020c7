"""CPU oracle for the tree-verification hot path — TEST INFRASTRUCTURE ONLY.

A plain, slow, deliberately literal restatement of what each step of the hot path
computes, written from the source pages and sharing no code with the CUDA library
(no kernels, headers, helpers, tables or pre/post-processing). Only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may import it; the product path never does.

Pages cited in this package (by title):
  [TRT]   "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿——三层隐状态、
          草稿循环与动态树验证"
  [HB]    "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE"
  [EAGLE2] the EAGLE v2 dynamic-tree walkthrough ("动态树解码 … initialize_tree /
          topK_generate / tree_decoding / evaluate_posterior"), sections 3-5.
  [MO]    "EAGLE头结构深潜: Model Optimizer 投机解码草稿模型的内部设计"

Precision: fp64 everywhere, except where a floating-point value decides an integer
(the joint top-k and the final selection): there the scores are held in fp32, the
precision the GPU path takes those decisions in, with each log-probability rounded
once to fp32 from an fp64 log-sum-exp.

Modules:
  tree       ancestor mask, depths/positions, retrieve_indices, child/sibling links
  draft      per-row log-softmax + top-k, joint pruning, final total_tokens selection
  attention  RoPE and tree-masked attention over the materialised T x (P+T) mask
  accept     greedy walk (handbook form), evaluate_posterior (EAGLE-2 form), KV compaction
  lm_head    the target's greedy token at every node (argmax of the lm_head logits)
  sampling   non-greedy acceptance: filtered target probabilities, tree rejection walk
  step       one whole hot-path pass for one request (used for the CPU baseline)
"""
from . import tree, draft, attention, accept, lm_head, sampling, step  # noqa: F401
