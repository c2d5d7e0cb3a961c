"""CPU oracle for attention-guided KV selection — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the hot path computes,
in fp64 numpy (fp32 only where the pages or the documented reading fix fp32).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import it.  The product path (the C-ABI library and
its Python binding) never imports, calls or links anything in here, and the
oracle shares no code with it.

Sources (web pages, cited by title and section):

* "Sparse attention x KV-cache offloading: eight questions" (p1)
  §1 (decode reads the whole KV every step), §2.1 (temporal aggregation),
  §3.1 (token->block aggregation: max / mean / top-p%), §3.2 (per-request
  percentile normalisation), §5.1 (fp32 score + int32 timestamp per block).
* "From sliding window to attention-guided eviction" (p2)
  §1.1 (KV growth, Llama-2-70B shape), §3.1 (softmax over all visible keys),
  §4.1 (StreamingLLM sink + window), §4.2 (H2O cumulative score and its
  pseudocode), §4.3 (SnapKV observation-window vote, max-pool, top-k, GQA).
* "Long context, KV eviction and sparse attention" (p3, handbook chapter)
  "The cost of long context" (KV bytes closed form and its printed output),
  "KV eviction: StreamingLLM" (keep rule for recent-only and sink+window),
  "Sparse attention: dynamic selection" (masked softmax, exact top-k, Quest
  page bound, relative-error metric) and the DSA lightning-indexer paragraph.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, library routines, brute force or values
printed on the pages.  No function is "parity unpinned".
"""
from . import attention, h2o, snapkv, block_priority, dsa, costs  # noqa: F401
