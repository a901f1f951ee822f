"""Reference oracle for the RadixAttention hot path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct CPU restatement of what the
hot path computes, written in Python + numpy float64 from the pages on
SGLang's RadixAttention.  It exists to check the CUDA library; it is never on
the product path.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import it.  It shares no code with the
library (no headers, helpers, tables or constants); both sides receive the
same inputs from the seeded generators in ``workloads/``, which hold none of
the method's arithmetic.

Modules
-------
tree       per-page trie (per-token when page_size == 1) with longest-prefix
           match, insert, ref-count lock/unlock, leaf-first LRU eviction and
           the free-list slot allocator; ``build_batch`` emits req_to_token.
groups     prefix groups (segments of positions shared by a set of requests)
           defined directly from the slot table.
attention  decode / extend attention as naive softmax over gathered slots,
           the log-sum-exp merge, and the shared-aware decode that computes
           each shared segment once.
kvbytes    the KV-bytes-per-token formulas (GQA and MLA) used for the roofline.
fp8        E4M3 decoding and dequantised views of FP8 pools.
sched      the round-based cache-aware scheduling simulation.
mla        MLA decode attention in the latent space (one stored row per
           token, read as key and, its latent prefix, as value).

Every function is pinned by ``tests/test_oracle_*.py`` against facts the
pages or the mathematics fix (brute force, closed forms, worked examples,
library special cases).
"""

from . import tree, groups, attention, kvbytes, fp8, sched, mla  # noqa: F401
