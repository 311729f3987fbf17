"""Plain, slow, obviously-correct CPU oracle for the block-sparse attention path.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference arm of ``bench.py`` may import it. The product
(``load_balancing_gb300``) never imports, calls or links anything here, and this
package imports nothing from the product.

Every floating-point result is computed in fp64 with numpy; integer work is done
with exact Python/numpy integers. Each function cites the passage of the source
pages it restates. The pages are:

* "db-SP：稀疏注意力头并行和序列并行的负载均衡问题" (db-SP load-balancing blog,
  yjmstr.github.io, 2026-01-30) -- cited as *db-SP blog*, with "scenario 1" (head
  balancing, LPT, its counter-example and its bound) and "scenario 2" (Q-/KV-block
  loads, Q-block rebalancing with a stay-in-place bonus, per-iteration KV greedy).
* "6D 并行下的 Attention Kernel 与通信重叠" (walkerchi.com study notes) -- cited as
  *6D attention notes*, §2.1 (ring-attention pseudocode with the online-softmax
  merge) and §2.3 (causal skipping, striped attention).

Modules:
  loads      -- mask row/column/head sums (db-SP blog, scenario 2, load bullet)
  lpt        -- textbook LPT with stay bonus, brute-force optimum (db-SP blog,
                scenario 1 and scenario 2 bonus bullet)
  attention  -- block-sparse masked softmax attention, final and partial outputs
                (6D attention notes §2.1 step 2 and final division)
  merge      -- online-softmax merge of (O, m, l) partials (6D attention notes
                §2.1 step 3)

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` to
values the pages print, closed forms, library routines or brute force; none is
"parity unpinned".
"""

from . import loads, lpt, attention, merge  # noqa: F401
