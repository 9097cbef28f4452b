"""CPU oracle for the lookahead-decoding step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what one lookahead decoding
step computes ("Break the Sequential Dependency of LLM Inference Using
Lookahead Decoding", arXiv 2402.02057, as summarised on the paper-graph-ui
page, section 3.4).  It is written in numpy, in float64 by default, and shares
no code with the CUDA path: neither imports the other.  Only the seeded input
generators in `synth` serve both.

Who may use it: the tests, `__graft_entry__.smoke()` and the CPU-baseline legs
of `bench.py`.  The product path never routes through it.

Modules
  decoder    -- LLaMA-style decoder forward with an explicit visibility matrix
  lookahead  -- step rows and mask, n-gram pool, greedy and sampling
                verification, window harvest/shift, AR and lookahead generation
  philox     -- Philox4x32-10 for the sampling draws

Pins: every function here is checked by `tests/test_oracle_*.py` against
something other than itself (closed forms, library routines, brute force,
published known answers, the pages' invariants).  None is "parity unpinned".
"""
