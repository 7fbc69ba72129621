"""CPU oracle for the DFlash drafting round -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of one DFlash drafting-plus-
acceptance round.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run anything in this package; the
product path (the CUDA library and its Python binding) never does.  It shares
no code with the CUDA path; its only shared dependency is the ``workload``
package of seeded input generators.

Pages it follows (cited by title and section throughout):
  [Code walkthrough]  "DFlash原理深度剖析：块扩散如何用一次前向并行起草整块token"
                      (kkqc.cn) -- sections 二.1, 二.2, 二.3, 三
  [Paper walkthrough] "DFlash：drafter 的答案，早写在 target model 的隐层里"
                      (bowenzhou.top) -- "Why DFlash?", "设计" (Feature Fusion,
                      KV Injection, Parallel Drafting)
  [News summary]      "DFlash：块扩散草稿模型实现最高15倍吞吐量提升"
                      (news.paixiangai.cn) -- "“目标模型最懂”的洞见"
  [NVIDIA blog]       "Boost Inference Performance Up to 15x on NVIDIA Blackwell
                      Using DFlash Speculative Decoding" -- "DFlash 预测解码的工作原理是什么？"

Parity status per function: every function below is pinned by the CPU tests
in tests/test_oracle_*.py except the absolute values of hidden states, logits
and K/V at realistic sizes, which nothing outside the oracle fixes
("parity unpinned" beyond the invariants and library cross-checks listed
there; the pages print no worked numeric example).
"""
from .dflash_ref import (  # noqa: F401
    bf16_to_f64,
    rmsnorm,
    rope,
    silu,
    softmax,
    fuse_features,
    inject_kv,
    block_attention,
    decoder_layer,
    lm_head_logits,
    argmax_first,
    accept_longest_prefix,
    synthetic_target,
    OracleModel,
    OracleRequest,
    OracleDrafter,
)
