"""CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, fp64 restatement of what the paged KV-cache
hot path computes, written from the source pages:

  * "external-cannbot-model-model-infer-kvcache" (KVCache Optimization Skill,
    Ascend cann-recipes-infer): Mode 2 (paged attention + FA), Mode 3 (MLA
    compressed cache), In-depth Principles 3.1-3.6, Appendices C and E.
  * The ai6s.net article on KVCache on Ascend NPUs: section 3 (cache size
    formula and its worked examples) and section 4 (CacheManager allocation,
    ND layout, and the KVCache write loop).
  * The hotelren.com source-reading notes "Paged KV Cache + Packed Sequence":
    sections 1.1, 2.1-2.3, 3.1-3.3, 4.1, 4.3 and 5.1.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The product package never imports it and shares
no code with it: the CUDA path has no CPU fallback.

Every function here is pinned by ``tests/test_oracle_pins.py`` and
``tests/test_oracle_bruteforce.py`` to values the pages print, to closed
forms, to invariants, or to an independent pure-Python brute force.
"""

from . import kvc_oracle, bruteforce  # noqa: F401
