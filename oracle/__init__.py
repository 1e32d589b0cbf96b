"""Oracle for the HiSparse RESOLVE hot path -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct CPU model that the CUDA
path is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  The product path (the
``host_offload_serving_gb300`` package and its C-ABI library) never imports,
links or calls anything here, and nothing here imports the product path.

Modules
-------
``tiny``        pure-Python model (``dict`` page table + explicit ``list`` LRU),
                plus a brute-force optimal (Belady) miss count for tiny traces.
``hisparse_oracle.c`` / ``coracle``
                the same definition written in plain single-threaded C, for
                the full-size workloads and for the timed CPU baseline.

Sources (cited by page title and section):
  [P1] gentlecold.top, "HiSparse 深度解析：论文、SGLang 实现与 vLLM Hybrid
       HiSparse" -- §3.3 (replacement policy), §3.4 (request lifecycle,
       write-through), §3.5 (RESOLVE fused kernel and its worked example),
       §3.6 (exact cross-layer prefetch), §5.2 (per-request tensors),
       §5.5 (swap-in kernel), §5.6 (prefetch in SGLang).
  [P5] notes.kuangjux.top, "HiSparse：稀疏注意力的分层 KV Cache 管理" --
       §5 (the {1,4,8}/{1,5,8}/{1,4,8} cache-capacity example).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked examples, textbook-LRU reduction, brute-force optimal bound,
invariants, closed forms).  No function is "parity unpinned".
"""
