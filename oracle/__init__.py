"""CPU oracle for paged serving attention -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.  The library (`serving_attention_plan_gb300`) never
imports it, and it shares no code with the library: the two meet only in the
seeded input generator (`serving_attention_plan_gb300.workloads`), which holds
no attention arithmetic.

Citations name the page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎"
(a digest of the MLSys 2025 paper "FlashInfer: Efficient and Customizable
Attention Engine for LLM Inference Serving") by its section headings, with the
paper section, algorithm or figure the page itself gives.

Modules
  attention -- float64 gather of BSR pages + softmax(q k^T * scale + mask) v and
               LSE, and the attention-state merge operator.  Every function is
               pinned by tests/test_oracle_attention.py (brute force, library
               special cases, closed forms, invariants).
  planner   -- the load-balancing plan restated in plain Python (lengths, tile
               choice, KV chunk bound, chunking, cost, longest-first assignment
               through a CTA priority queue, reduction map).  Pinned by
               tests/test_oracle_planner.py (a hand-worked plan, coverage
               invariants, the partial-output bound, Graham's LPT bound against
               brute-force optimal makespans).
"""
