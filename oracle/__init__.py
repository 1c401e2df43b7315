"""Plain, slow, CPU reference ("oracle") for sparse-graph attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package: only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
it. It shares no code with the CUDA library; the only common module is ``workloads``
(seeded input generators, no method arithmetic).

Everything is numpy float64 (integers for masks), written to be checked by eye
against the pages it follows:

* [CAS] "Parameter-free Adaptive Sparse Attention via Compression-Based Content
  Selection" (arXiv 2607.21752): per-block gzip ratio (section 3.1, Eq. 1), mean
  threshold (Eq. 2), block mask of literal pairs, local window and identity
  (section 3.2, Eq. 3; Appendix B, Algorithm 1), block-to-token expansion with causal
  intersection (section 3.4).
* [BB] "BigBird" (llm-arch-kb, section 2 "Derivation" and section 3 "Reference
  implementation"): window, global and random sub-graphs and their edge counts.
* [FIB] "Depth-Staggered Fibonacci Spacing for Sparse Attention" (arXiv 2606.28560,
  section 2 "Method"): dense window {0..W} plus offsets d_k = alpha * f_k.

Readings taken where the pages are silent or disagree are stated at each function. Parity status: every function here is pinned by ``tests/test_oracle_*``
against closed forms, brute force from the token-level definitions, library routines
(numpy's Philox, gzip framing) or an independent dense route.
"""
from .ratios import block_ratios, zlib_version
from .philox import philox4x64_10, philox_word
from .masks import (MaskParams, build_csr, csr_topk_rows, csr_bigbird_rows, csr_full_rows,
                    csr_literal_mean_rows, csr_to_block_mask, block_mask_to_token_mask,
                    literal_flags, topk_row_count, cas_head_components, LOCAL, LITERAL)
from .fib import (fib_rungs, fib_rungs_upto, pow2_rungs, pow2_rungs_upto, alpha_schedule, fib_offsets,
                  offset_key_set, interp_rungs)
from .attention import (attention_csr, attention_csr_block, attention_csr_heads, attention_offsets,
                        dense_masked_attention, attention_rows_csr, attention_csr_backward, attention_rows_dq,
                        attention_rows_dkdv, attention_offsets_interp, attention_csr_backward_heads)

__all__ = [
    "block_ratios", "zlib_version", "philox4x64_10", "philox_word", "MaskParams", "build_csr",
    "csr_topk_rows", "csr_bigbird_rows", "csr_full_rows", "csr_literal_mean_rows",
    "csr_to_block_mask", "block_mask_to_token_mask", "literal_flags", "topk_row_count",
    "cas_head_components", "LOCAL", "LITERAL", "attention_csr_heads",
    "fib_rungs", "fib_rungs_upto", "pow2_rungs", "pow2_rungs_upto", "alpha_schedule", "fib_offsets", "offset_key_set", "attention_csr",
    "attention_csr_block",
    "attention_offsets", "dense_masked_attention", "attention_rows_csr", "attention_csr_backward",
    "attention_rows_dq", "attention_rows_dkdv", "attention_offsets_interp", "interp_rungs",
    "attention_csr_backward_heads",
]
