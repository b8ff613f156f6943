"""CPU oracle for paged MLA decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (``paged_mla_decode_10_gb300``)
never imports it, and this package never imports the product library.

* :mod:`oracle.reference` -- the fp64 C implementation of the decode
  (``mla_oracle.c``) behind a ctypes wrapper.
* :mod:`oracle.metadata` -- the split-KV schedule written out as a plain
  Python walk, and a checker of the invariants every schedule must meet.

Parity status: the decode function is pinned by closed forms, invariants and
a dense library routine (see tests/test_oracle_*.py); the schedule walk is a
restatement of a policy this library chose (the pages leave it open), pinned
by the coverage invariants.
"""
