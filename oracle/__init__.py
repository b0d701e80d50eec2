"""Float64 CPU oracle for the gated delta rule (TEST INFRASTRUCTURE ONLY).

This package is the yardstick the CUDA path is measured against. It is
plain, slow and written to be checked by eye against the pages it cites:

* ``recurrence``  -- the token-by-token recurrences, one per page and in
  each page's own state orientation, plus the unified form all four
  variants share (numpy, fp64, one sequence at a time).
* ``chunked``     -- the chunkwise WY/UT algebra exactly as the
  Gated DeltaNet-2 notes state it (numpy, fp64, no blocking beyond the
  chunk the algorithm itself defines).
* ``expansion``   -- the closed-form product expansion of the affine
  recurrence (LLMs-from-scratch ch. 11, section 11.4).
* ``backward``    -- gradients: float64 autograd through the token recurrence,
  and the chunkwise backward of the Gated DeltaNet-2 notes (key design 3).
* ``epilogue``    -- the output epilogue after the read-out: RMSNorm over
  the value channels times a gain, then the SiLU output gate (numpy, fp64).
* ``native``      -- a ctypes wrapper around ``gdr_oracle.c``: the same
  unified token recurrence in plain C (fp64, OpenMP over heads) for the
  sizes numpy cannot finish, and for the timed CPU baseline.

Who may use it: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``. The product
path (the ``gated_delta_rule_10_gb300`` package and its CUDA library)
never imports, links or executes anything here, and nothing here imports
the product package: the two share no code. Seeded inputs come from
``gated_delta_rule_10_gb300.workloads``, which holds no arithmetic of the
method and is passed in by the caller.

Every function states the passage it follows. Functions without an
independent pin say "parity unpinned" in their docstring; at present the
only such reading is the choice of which query vector enters Q-Delta's
mixed erase input (see ``recurrence.qdelta_q_delta_page``).
"""
