"""CPU oracle for the paged latent-cache path -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline leg
(and its ``--impl reference`` arm) may import, call, link or execute anything
in this package.  The product library never does, and the two share no code:
the oracle imports nothing from ``paged_mla_kv_gb300``.  Both sides take their
inputs from the seeded generator module ``paged_mla_kv_gb300.synth``, which holds
no method arithmetic; the tests hand those inputs to the oracle.

Modules:
  attend  -- attention over contiguous latent rows (and over listed rows) in fp64 (C, via ctypes)
  fp8     -- E4M3 codes from their bit fields, per-row quantization and dequantization
  paged   -- expected pool images after appends and kept-state copies
  plan    -- the kv_pool plan arithmetic in integers
  topk    -- the top-k of a row under the IEEE total order, and its blocked form
  build   -- compiles the C part with gcc

Parity status: every function here is pinned by tests/test_oracle_*.py against
closed forms, special cases that reduce to library routines, brute force on
tiny inputs and the pages' worked numbers; none is "parity unpinned".
"""
