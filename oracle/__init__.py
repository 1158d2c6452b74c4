"""CPU oracle for paged decode attention — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct reference code.  Only the test suite, the
package's ``__graft_entry__.smoke()`` check and the benchmark's CPU-baseline /
reference arm may import or run anything in this package.  The CUDA library
never imports it and shares no code with it.

Contents
  block_manager  refcounted block manager (allocate / free / fork /
                 blocks-needed / append / physical index) plus copy-on-write
  attention      fp64 decode attention over a paged KV pool
  cache_ops      byte-exact cache write (reshape_and_cache) and block copy
  brute          pure-Python loops for tiny cases (math.exp, no numpy)
  scenarios      the decode workloads' pool layouts, built through the
                 block manager from a seed
  accounting     KV byte arithmetic (bytes per token, sharing savings)

Every function cites the page and section it follows.  The four source pages
are referred to as:
  "PagedAttention" glossary entry (inferensys.com)
  "10 — Paged Attention" tutorial (infra.pidoku.co.in, v-llm-inference)
  "PagedAttention: Virtual Memory for KV-Cache" (insidellms.com, ch. 4.4)
  "PagedAttention & KV-Cache Management in High-Throughput LLM Serving"
      (subroutine-cs.cc)

Parity status: every function here is pinned by a ``-m "not gpu"`` test
against something other than itself (a traced worked example, closed forms,
a library attention routine over contiguous storage, invariances, brute
force).  No function is parity-unpinned.
"""
