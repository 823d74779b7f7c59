"""Float64 CPU oracle for paged MLA decode — TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct reference that the CUDA path is checked
against. It is not part of the product: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s ``cpu_baseline`` / ``--impl reference`` legs may import it. The
library in ``mla_paged_decode_02_gb300`` never imports it, and it never imports the
library; the two share no code. The only module both sides use is the seeded input
generator ``mla_paged_decode_02_gb300.synth``, which holds no attention arithmetic.

Modules
-------
fp8_e4m3    OCP FP8 E4M3 ("fn" variant) decode table and round-to-nearest-even,
            saturating encoder.
mla_oracle  Cache write, page-walking gather, absorbed-MQA decode, split/LSE combine
            and the kernel test's cosine-difference metric.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against
something other than itself (torch's float8 conversion, a brute-force nearest-code
search, a pure-Python loop decode, torch's scaled_dot_product_attention, and
invariants). No function is "parity unpinned".
"""
