"""CPU oracle for the drafter head and the speculative verifier.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The CUDA library never calls it, and
it shares no code with the library: it is a plain, slow restatement, in numpy
float64 (exact rationals where a test asks for them), of what the articles say
the path computes.

Sources (each function names the one it follows):

* "SlimSpec article" -- 荷兰Nebius团队：给AI“起草员“瘦身，大模型推理速度提升5倍
  (mhpn.cn).  Section 三 defines the low-rank head (W_down: d -> r, W_up: r -> V,
  cost O(r*d + V*r), r = d/8); section 四 the acceptance rate sum_x min(p, q);
  section 二 static vocabulary trimming (FR-Spec, VocabTrim).
* "SpecVocab write-up" -- 动态词汇推测加速大语言模型推理 (2kiu.com).  Sections
  2.2.1-2.2.3: h' = W_down h at d' = d/16, s = W_vocab h', k_t = topk(s, 2048),
  z' = U[k_t] h, q = softmax(z').  Section 3.3: verification still uses the full
  vocabulary.
* "Explainer" -- 大模型批改 5 个词，和自己写 1 个词一样快：投机解码讲人话
  (liuchunshan.com).  Section "小模型起草，大模型批改": verify left to right, keep
  the matching prefix, replace the first mismatch by the target's token, one
  extra target token when all match.  Section "为什么答案不会变": greedy keeps
  only target-argmax tokens; sampling accepts with probability min(1, p/q),
  resamples a rejection from the renormalised positive part of p - q, and the
  output distribution equals p exactly.  Section "这笔账划不划算，看一个数":
  the closed form for expected tokens per round and its table at gamma = 4.
* Salmon, Moraes, Dror & Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
  (SC'11), section 4: the Philox4x32-10 counter-based generator that both
  sides draw their uniforms from when the caller passes a seed and an offset
  instead of its own uniforms.
* "SpecTr-GBV article" -- SpecTr-GBV: Multi-Draft Block Verification
  (hypresin.com), 第三步: residual draw when the accepted block is short of the
  full length, one extra target token when the whole block is accepted.

Readings taken where the articles are silent:
  * W_down is stored r x d and applied as h @ W_down.T.
  * The intermediate z (and SpecVocab's h') is rounded to nearest-even bf16 for
    bf16 workloads; fp32 workloads keep it unrounded.
  * Ties in argmax, top-k and inverse-CDF go to the lowest vocabulary index.
  * Sampling uses one uniform u per draw (the caller's own, or Philox4x32-10
    at the draw's (seed, offset, row, slot) counter) and inverse-CDF over the
    weights in ascending vocabulary order.
  * Temperature divides both target and draft logits.
  * An all-zero residual falls back to p at that position.

Pinning: every function here is checked by ``tests/test_oracle_*.py`` against
closed forms, the articles' printed values (``tests/golden``), library routines
and exact enumeration.  No function is "parity unpinned".
"""
from .bf16 import round_to_bf16
from .head import down_projection, up_projection, dense_logits, row_reduce, \
    inverse_cdf, slimspec_head, dense_head, trimmed_head
from .specvocab import approx_scores, topk_lowest_index, specvocab_head
from .verify import softmax_t, verify_greedy, verify_decide, verify_sampling, verify_batch, \
    verify_lowrank_batch
from .philox import philox_block, philox4x32_10, uniforms as philox_uniforms
from . import theory

__all__ = [
    "round_to_bf16", "down_projection", "up_projection", "dense_logits",
    "row_reduce", "inverse_cdf", "slimspec_head", "dense_head", "trimmed_head", "approx_scores",
    "topk_lowest_index", "specvocab_head", "softmax_t", "verify_greedy",
    "verify_decide", "verify_sampling", "verify_batch", "verify_lowrank_batch", "theory",
    "philox_block", "philox4x32_10", "philox_uniforms",
]
