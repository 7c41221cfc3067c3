"""CPU oracle for the packed-THD attention hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import this package; the product path never
does, and this package imports nothing from the product path.

Everything here is a plain, slow, obviously correct restatement of what the
pages define, in float64 on the same bf16-rounded inputs the GPU sees:

* ``attention``  exact softmax attention with the segment/causal/window mask
                 ("Context parallelism and ring attention", section "The
                 attention problem"; TE tutorial section 3 "Fused attention
                 call"), its LSE, the exact valid-pair count, and the
                 explicit-P gradient.
* ``merge``      the (m, z, u) running-softmax update of section "Online
                 softmax".
* ``reorder``    the causal load-balancing permutations (section "Load
                 balance"; TE tutorial section 4).
* ``plan``       per-tile SKIP / FULL / PARTIAL classification (section
                 "Causal attention").
* ``ring``       ring attention over R logical shards (section "Ring
                 attention").
* ``brute``      pure-Python triple-loop attention for tiny inputs.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_*.py``; none is "parity unpinned".
"""
