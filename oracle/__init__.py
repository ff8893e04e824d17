"""Plain fp64 CPU oracle for the SparseVILA hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only the test suite, the package smoke check and the CPU-baseline leg of the
benchmark may call it.  It shares no code with the CUDA library and never
imports it.

Every function restates the definition given on the SparseVILA pages in the
plainest way, in float64, with no blocking, fusion or reordering beyond what the
definition states.  The pages (all describing "SparseVILA: Decoupling Visual
Sparsity for Efficient VLM Inference", arXiv 2510.17777) are cited by site and
section:

* velog.io summary -- §3.1 Prefill Phase (query-agnostic pruning, salience
  table, kernel), §3.2 Decode Phase (query-aware retrieval, dense packing),
  §4.1 Setup (partial KV-cache eviction, sparsity policy).
* xllm-io review -- §三 "核心公式" (salience and retrieval formulas) and §五
  "代码实现分析" (prune / retrieve / evict procedures).
* sciencestack.ai abstract page -- abstract and Figure 4 caption.

Pin status: every function here is pinned by CPU tests (closed forms,
invariants, brute force on tiny inputs, library routines); none is
"parity unpinned".
"""

from .sparsevila import (  # noqa: F401
    BLOCK_TOKENS,
    salience,
    summary_salience,
    topk_ascending,
    prune_compact,
    prune_threshold,
    paged_view,
    retrieval_scores,
    retrieve_topk,
    retrieval_scores_softmax,
    sparse_decode_attention,
    pack_selected_kv,
    evict_qa_tokens,
    append_tokens,
)
