"""CPU oracle for paged MLA decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library (``paged_mla_decode_10_gb300``)
never imports it, and this package never imports the product library.

* :mod:`oracle.reference` -- the fp64 C implementation of the decode
  (``mla_oracle.c``) behind a ctypes wrapper.
* :mod:`oracle.metadata` -- the split-KV schedule written out as a plain
  Python walk, and a checker of the invariants every schedule must meet.
* :mod:`oracle.fp8` -- the decode over an e4m3 query and latent cache with
  the two fused product scales: an e4m3 decoder written from the format's
  bit layout, in front of :mod:`oracle.reference`.

Parity status: the decode function (bf16 and e4m3) is pinned by closed forms,
invariants and a dense library routine (see tests/test_oracle_*.py); the
e4m3 decoder by torch's float8_e4m3fn conversion; the schedule walk is a
restatement of a policy this library chose (the pages leave it open), pinned
by the coverage invariants.
"""
