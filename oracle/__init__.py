"""fp64 CPU oracle for masked scaled-dot-product attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product (``long_context_masked_mask_gb300``) never
imports it and shares no code with it; the only module both sides use is
``synthetic`` (seeded random draws, no arithmetic of the method).

What it follows: the pages ("Long-Context Attention Benchmark: From Kernel
Efficiency to Distributed Context Parallelism"; xllm-io blog review, sections
"注意力掩码模式" and "密集注意力内核") name the operator every benchmarked kernel
computes -- masked softmax attention, forward and backward, bf16, head dim 128,
MHA and GQA -- and fourteen mask families by name only.  The pages print no
formula, so the oracle writes out the textbook definition:

    S = s * Q K^T,  P = softmax over the allowed keys of each row,  O = P V,
    LSE_i = log sum_{j allowed} exp(S_ij)

and its gradients for L = <O, dO>.  Mask predicates are the plain readings of
the mask names (see ``masks_ref``).  ``block_select_ref`` writes out the step
that produces a dynamic block map -- TopK / TopP selection of key blocks from
pooled Q K^T scores, the criterion the paper's peer reviews name (tomesphere
page, section "Peer Reviews") -- under the readings stated in its docstring.

Pins (tests/test_oracle_*.py): torch's own fp64 scaled_dot_product_attention
and autograd on tiny cases, central finite differences, closed forms (N = 1,
uniform keys), row sums, hand-derived small masks and block selections in
``tests/golden``, brute force over every subset for TopK / TopP, the
bilinearity identity for pooled scores, and the invariants between mask
families and selection parameters.  Every function here is pinned; none is
"parity unpinned".
"""
from . import block_select_ref, fp8_ref
from .masks_ref import allowed, allowed_pairs
from .attention_ref import (attention_fwd, attention_bwd, attention_fwd_rows, attention_bwd_rows,
                            attention_bwd_sampled, classify_tiles, EMPTY, FULL, PARTIAL)

__all__ = ["block_select_ref", "fp8_ref", "allowed", "allowed_pairs", "attention_fwd", "attention_bwd", "attention_fwd_rows",
           "attention_bwd_rows", "attention_bwd_sampled", "classify_tiles", "EMPTY", "FULL", "PARTIAL"]
