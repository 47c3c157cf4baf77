"""CPU oracle for the tree-verification step: test infrastructure only.

A plain, slow, obviously-correct restatement of what the step computes,
written from the pages' statement of the method (numpy, float64 unless a
decision is stated to be taken in the kernel's float32).  It shares no code
with the CUDA path: it reads the same seeded inputs (from the package's
``synth`` module, which holds none of the method's arithmetic) and nothing
else.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
cpu-baseline / reference leg may import it; the product path never does.

Modules
-------
tree       depth, ancestor mask, depth-based position ids, child links,
           static (Medusa) token placement, confidence-product rerank
heads      Medusa residual heads, LM head, top-s selection
attention  tree attention, explicit per node over prefix + ancestors
accept     greedy / typical / rejection acceptance and the bonus token
commit     copy of the accepted path's K/V rows into the cache
expand     one confidence-product expansion round (EAGLE-2 style)
expected   expected accepted length (closed forms on the pages)
rng        Philox4x32-10 counter-based generator

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` (worked values printed on the pages, textbook
special cases, brute force, exact enumeration); none is "parity unpinned".
"""
