"""fp64 CPU oracle for tree-structured speculative verification of gated-DeltaNet hybrids.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never imports, calls or links it, and this package
imports nothing from the product path: the two share no code.  The only module both sides
use is ``workloads``, the seeded input generator, which holds none of the method's
arithmetic.

Plain, slow and meant to be checked by eye against the pages: numpy in fp64, loops over
sequences, nodes and heads, no blocking or fusion.

* ``tree``      -- depth, tree mask, root-to-node paths, validity.
* ``gdn``       -- gated delta rule per node by path replay; the depth-by-depth schedule;
                   TreeWY pseudo-values from their definitions; commit.
* ``attention`` -- RoPE, dense masked-softmax GQA attention over a paged prefix, cache
                   writes, KV compaction.

Every function is pinned by a CPU test against something other than itself (a printed
example, a closed form, a library routine, an invariant or brute force): see
``tests/test_oracle_*.py``.  No function is unpinned.
"""
from . import attention, gdn, tree  # noqa: F401
