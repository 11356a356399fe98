"""Oracle for the Momentum DeltaNet (MDN) memory update — TEST INFRASTRUCTURE.

Plain, slow, fp64 CPU implementations of what the CUDA path computes, written
from the MDN paper-reading slides and the MDN reading notes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and
``--impl reference``) may import anything from here.  The product path
(``momentum_delta_rule_gb300``) never imports, links or calls this package,
and this package never imports the product.

Contents
  recurrence   fp64 token-by-token recurrence (C, OpenMP) — the parity oracle
  coefficients fp64 chunk coefficients in four independent forms
  chunkwise    fp64 chunkwise-parallel forward (Gamma, shifted Gamma, solve)
  backward     fp64 gradient of the recurrence (reverse sweep over states
               rebuilt from the saved residuals), for the backward pass
  chunkwise_backward  fp64 gradient of the chunkwise form (per-chunk dense
               products, state adjoints carried backwards across chunks)
  build        compiles the C oracle with gcc (building the checker is not
               using it)

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
what the pages and the mathematics fix (special-case reductions, the
two-step worked example, the block transition matrix and its spectrum, the
second-order identity, brute force on tiny inputs); each test names the
passage of the pages it follows.
"""
