"""Plain CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The library's product path (the CUDA kernels behind the C ABI and their Python
binding) never imports, calls or falls back to anything in this package.

Modules:
  spec_oracle  float64 NumPy restatement of the verification rules
               (greedy chain, stochastic chain, tree walk, residual,
               closed-form induced distribution).
  exact        exact-rational (fractions.Fraction) brute force of the whole
               speculative procedure on tiny vocabularies, used to pin
               spec_oracle against the losslessness the pages prove.

Parity status of each function is given in its module header.
"""
