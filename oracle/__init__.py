"""Float64 CPU oracle for fused dequant-on-load flash-decode over a quantized KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing here is part of the product: only the test suite,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import it.  The library under ``flash_decode_quantized_gb300`` never
imports it and shares no code, table or helper with it; the two meet only through the
documented byte layout of the store and through the seeded inputs of ``workloads``.

What the oracle computes, and where each piece comes from:

* ``codec``     -- the q8_0 and 4-bit symmetric block codecs (encode, pack, decode) and
                   the 16-bit control stores.  q8_0 is the KV type of the A/B in
                   "halobench record clm-0022" (METHOD and depth tables); 4-bit-V codecs
                   are named in rMLX issue #292 (symptom and correction tables).  Neither
                   page prints the arithmetic; the block rule used here (32 elements along
                   head_dim, fp16 scale d = amax/c, q = round(x/d), c = 127 or 7) is the
                   library's codec contract.
* ``store``     -- the paged, structure-of-arrays byte layout of a resident KV store
                   (the "keep the prefix resident on-device" fix direction of rMLX issue
                   #295, "Fix direction").
* ``attention`` -- single-token softmax attention with grouped query heads, plus the
                   split-K (m, l, acc) partial/combine form of flash-decode (rMLX issue
                   #292, "Root cause": the flash-decode-over-quant kernel class).

Parity status of every function is stated in its docstring ("pinned by ..." or
"parity unpinned").
"""

from . import codec, store, attention  # noqa: F401
