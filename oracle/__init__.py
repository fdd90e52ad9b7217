"""CPU oracle for starting-node triangular self-attention: test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the product path never does.
"""
