"""CPU oracle for tree-attention speculative verification — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the verification step
computes, in fp64 (numpy) with pure-Python loops where the inputs are small.
It exists so that the CUDA library can be checked against an independent
definition.  Only the test-suite, the smoke check and the benchmark's CPU
baseline leg may import it; the library itself never does, and it shares no
code, table or helper with the CUDA path.  Inputs come from ``workloads``.

Sources (three web pages on the method):
  [P1] "Tree Attention" — inferensys glossary (sections: What is Tree Attention;
       Key Mechanisms: Batched Parallel Verification, Modified Causal Attention
       Mask, Speculative KV Cache Reuse, Multi-Token Acceptance & Rollback,
       Integration with Speculative Decoding).
  [P2] "Tree Attention" — zhongzhoutan-coder terms page (sections: How It Works,
       Tradeoffs, Common Confusions).
  [P3] "Speculative Tree Attention: How Multi-Candidate Draft Models and Parallel
       Verification Deliver 4x LLM Speedups" — premlal news (code listing:
       TreeNode, build_tree_attention_mask, verify_candidate_tree, demo;
       sections Production Inference Runtimes, The Future of Reasoning).

Modules:
  tree       — tree validity, ancestry mask by parent walk, depth, positions.
  attention  — masked softmax attention over prefix + ancestors, fp64.
  verify     — greedy argmax and the acceptance walk by definition.
  commit     — appending the accepted path's keys/values to the paged cache.
  stochastic — temperature verification by recursive rejection sampling.
  dynamic    — reranking a draft's candidate pool into the tree to verify.
  forest     — several roots in one flattened sequence: masks and acceptance.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
the pages' worked example, closed forms, library routines on special cases, or
brute force (see tests/test_oracle_*.py).  No function is "parity unpinned".
"""
from . import tree, attention, verify, commit, stochastic, dynamic, forest  # noqa: F401

# Status codes, restated here (the oracle shares no header with the library).
OK = 0
ERR_SHAPE = -2
ERR_BAD_TREE = -3
