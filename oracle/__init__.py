"""The oracle: a plain, slow, obviously correct CPU restatement of prefix-shared
decode attention (ChunkAttention), in float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only the test suite, the package smoke
check and the benchmark's CPU-baseline leg use it.  It shares no code with the
CUDA path (no kernels, headers, helpers, tables or constant generators); the
only module both sides use is ``workloads``, which draws seeded random inputs
and holds none of the method's arithmetic.

Sources (cited by page title and section throughout):

* "ChunkAttention: Efficient Self-Attention with Prefix-Aware KV Cache and
  Two-Phase Partition" (the arXiv 2402.15220v4 summary page), cited as
  [CA-summary §n].
* "ACL 2024論文解説: ChunkAttention — プレフィックスKVキャッシュ共有による
  マルチテナント推論高速化" (the explainer blog), cited as [CA-blog, <section>].

Modules:

* ``pakv``      the prefix-aware KV cache: a trie of fixed-size chunks with a
                 refcounted slot allocator [CA-summary §3.1; CA-blog,
                 Prefix-Aware KV Cache / 動的プレフィックス検出].
* ``schedule``  the per-step tables of the two-phase partition
                 [CA-summary §3.2, §3.3].
* ``fp8``       FP8 E4M3 quantisation of stored K/V for an 8-bit pool (the
                 published E4M3 format, restated from its definition).
* ``attention`` decode attention by its plain definition, the partial-result
                 triple (o, m, s) and its log-sum-exp merge, and the two-phase
                 evaluation over the schedule tables [CA-blog, Two-Phase
                 Partition; CA-summary §3.2].

Parity status: every function here is pinned by tests that do not call back
into the same arithmetic (brute force on tiny inputs, closed forms,
invariants, hand-derived table fixtures); none is "parity unpinned".
"""
