"""FP64 CPU oracle for the chunkwise gated delta-rule operator.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``. The product package never imports
it, and it shares no code with the CUDA library.

* ``recurrence`` -- ctypes wrapper of ``kda_oracle.c``: the token-by-token
  recurrence with hand-derived back-propagation through time (the definition).
* ``chunk_ref`` -- a numpy FP64 restatement of the chunk form (WY forward,
  ReWY and seven-product backward, matrix intra, Gram elimination). It pins the
  equations the pages lost in extraction against the recurrence and is a
  debugging aid; it is never the reference a GPU result is graded against.
* ``prologue`` -- numpy FP64 gate activation (softplus and lower-bound forms,
  with A_log and dt_bias) and q/k L2 normalisation, forward and backward;
  ``cases.run_oracle_prologue_arrays`` composes them with the recurrence.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against finite differences, closed forms, invariants and the pages' printed
counts. No function is "parity unpinned".
"""

from .recurrence import build, lib_path, run_recurrence  # noqa: F401
