"""CPU oracle for the sparse-attention indexer hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only the test suite, the smoke check and the benchmark's
CPU-baseline leg do.  It shares no code with the CUDA library; the only thing
both sides use is the seeded input generator module, which holds none of the
method's arithmetic.

Each function is a plain, slow, obviously correct restatement of a definition
or algorithm on the source pages, with the passage it follows in its docstring:

  dsa          indexer score s(k) = sum_h w_h ReLU(q_h . k) and exact top-K
               ("DoSA: ..." page, section 3 and section 1) -- fp64
  dosa         DoSA safe-upper-bound pruning, step by step in the page's order
               ("DoSA: ..." page, sections 2, 3.1, 3.2, 4) -- fp64
  witness      segment witnesses ("Segment Witnesses" page) -- integers
  block_select MiniMax block-max selection ("ferrox_core/block_sparse.rs"
               page) -- fp32 with the page's sequential dot order

Parity status: every function is pinned by the non-GPU tests against worked
examples printed on the pages, closed forms, invariants or brute force, except
the DoSA planning heuristics (choice of retained heads and anchors, the seed
rule), which the pages do not state; those are "parity unpinned" and only the
validity of the bound and the exactness of the output are pinned.
"""
