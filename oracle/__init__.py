"""Plain, slow CPU oracle for the paged KV cache hot path.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``;
nothing on the product path imports, calls or links it, and it shares no
code, header, table or helper with the CUDA library.  Its inputs are plain
NumPy arrays (or Python lists); the seeded generators that both sides use
live in ``paged_kv_cache_145_gb300/synth.py`` and hold none of the method's
arithmetic.

Modules
-------
``paging``     address translation and allocation accounting
``blocks``     reference-counted block pool with copy-on-write (host model)
``attention``  KV write, block copy and single-query attention in float64

Sources (web pages; cited by title and section in every docstring):

[vLLM-TGI]  "Inside vLLM and TGI: Paging, Versioned Schedulers and
            Operations" -- sections "Block addresses and fragmentation
            arithmetic" and "Exact CPU block manager and copy-on-write".
[VM-LLM]    "vLLM and PagedAttention: Virtual Memory for LLM Serving"
            (talk transcript; it has no headings, so paragraphs are named
            by topic: sizing, paging, sharing, preemption, results).
[CB-PA]     "Continuous Batching & PagedAttention: vLLM Memory Management
            Architecture" -- section "Core PagedAttention Mechanics".

Every function is pinned by ``tests/test_oracle_*.py`` to something other
than itself: values the pages print, closed forms, brute force on tiny
inputs, an independent library routine, or invariants.
"""

from . import paging, blocks, attention  # noqa: F401
