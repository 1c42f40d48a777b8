"""Float64 CPU oracle of the selective scan: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. Functions without a pin to the pages or
to mathematics are marked "parity unpinned" where they are defined; every
function here is currently pinned by ``tests/test_oracle_pins.py``.
"""
