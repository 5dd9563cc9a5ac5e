"""Reference oracle for the paged KV cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call or
execute anything in this package.  The product path (the CUDA library under
``paged_kv_cache_152_gb300/``) never imports it, and this package never imports
the product; the two share only the seeded input generators in ``workloads/``.

Everything here is plain, slow and written to be checked by eye against the
three web pages that define the method:

* [P1] "Paged Attention: OS-Inspired Memory Management for KV Caches"
  (modernaiengineering.com, lesson 13.6);
* [P2] "What is PagedAttention and how does it manage KV cache?" (n4n.ai blog);
* [P3] the worksonmygpu.com deep-dive post on PagedAttention in vLLM.

Floating point is fp64 throughout (the pages fix no precision); fp16 inputs are
upcast exactly.  Modules:

* ``attention``     -- decode attention through a block table, written as the
                       plain definition softmax(scale * q K^T) V over the tokens
                       gathered in logical order.
* ``cache_ops``     -- slot-mapped cache write and whole-block copy, as byte
                       copies.
* ``block_manager`` -- the block manager (free list, reference counts,
                       on-demand append, fork, copy-on-write, release).
* ``accounting``    -- block counts, slot waste and KV bytes per token.

Every function is pinned by ``tests/test_oracle_*.py`` to values the pages
print, closed forms, invariants or library routines.  No function here is
"parity unpinned".
"""

from . import accounting, attention, block_manager, cache_ops  # noqa: F401
