"""Oracle for the paged KV cache: plain, slow, obviously correct CPU code.

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its CPU-baseline leg and ``--impl reference``) may import, call,
link or execute anything in it. The product library (``paged_kv_cache_88_gb300``)
never imports it and shares no code, header, table or helper with it; the two meet
only in the seeded input generators of ``workloads``, which hold none of the
method's arithmetic.

Sources. The method is described by five web pages; the three that describe it are
cited by their address and their own section numbers:

* ``hnwysp.cn/news/103996`` -- KV-cache sizing, shared block pool, block table,
  refcount and copy-on-write, FIFO free queue (its sections 1.2, 3.1-3.5, 4.1-4.4).
* ``icman.com.cn/news/78786`` -- PagedAttention: block size and waste, pool
  arithmetic, paged attention kernel, prefix sharing (its sections 1.1-6.5).
* ``m.lqnn.cn/news/240480`` -- "kvcache sharemem": page pool, page table, index
  remapping inside the attention kernel (its sections 3.1-3.3, 5.2).

Modules:

* ``sizes``     -- closed-form KV sizes, pool arithmetic and internal waste.
* ``ref_alloc`` -- block pool: FIFO free queue, refcounts, append-slot and COW.
* ``ref_attn``  -- gather-then-attend decode attention in float64, the append
  scatter and the block copy (NumPy).
* ``ref_attn_c``-- the same attention definition in plain C (float64, OpenMP over
  (sequence, head)); the timed CPU baseline. Built by ``oracle.cbuild``.

Parity status of every function is pinned by ``tests/test_oracle_*.py``.
"""
