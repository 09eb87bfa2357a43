"""CPU oracle for the RESOLVE step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the smoke check in ``__graft_entry__`` and the benchmark's
CPU-baseline / reference leg may import this package.  The product path (the
CUDA library and its Python binding) never imports it and fails loudly when
its own extension is missing.

Modules:
  ``oracle.oracle``     -- ctypes driver of the C LRU simulator
                           (``hs_oracle.c``);
  ``oracle.attention``  -- float64 sparse attention over selected records,
                           for the exactness check.

Pins (tests that tie the oracle to something other than itself):
  ``Pair.resolve`` / ``Pair.run`` -- hand-worked trace, exhaustive and random
      brute-force replay, closed-form special cases, invariants, rejection
      of invalid selections (tests/test_oracle_pins.py);
  ``Pair.prefetch_plan`` / ``Pair.prefetch_copy`` / plan consumption --
      final state with a plan equals the state without one, for exact and
      for corrupted plans (tests/test_oracle_properties.py);
  ``attention.sparse_attention`` -- a one-hot layout check and equality with
      attention over the host records (tests/test_oracle_properties.py).
  The miss-rate values of the pages' own trace are parity unpinned: that
  trace is not available, only the direction (B = k misses more than
  B = 2k) is checked.
"""
