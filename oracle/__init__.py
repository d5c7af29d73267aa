"""Plain, slow, fp64 CPU oracle for batched draft verification.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or constants) and imports nothing
from it.

Modules
-------
``verify``        the verification rules themselves (chain, tree, cascade),
                  written step by step in float64 NumPy, one sequence at a time.
``closed_forms``  the PipeSpec analytical model (expected tokens per step,
                  steady-state verification probability and its recurrence).
``compact``       the cache compaction after a tree verification (the kept
                  root path's rows moved to contiguous positions).
``pipeline``      the k-model PipeSpec snapshot (stages 1 .. k-1, rollback of
                  every earlier buffer, an optional final-stage bonus).
``consulted``     the chain rule consulting rows in position order (rows after
                  the first rejection are never read).
``clasp``         the CLaSp layer-selection dynamic program and its
                  backtracking, on synthetic residual layers.
``lm_head``       chain verification from the final hidden states and the
                  LM-head weights (the logits as exact products).
``consulted_tree`` the tree walk consulting only the rows of the nodes it
                  visits (rows off the path are never read).
``pipeline_async`` the PipeSpec stages at independent buffer offsets (each
                  stage a chain verification of its own window, then the
                  rollbacks).

Every function states the passage it follows.  Points where the pages are
silent or ambiguous follow the readings listed in the design notes; each is
repeated in the docstring that depends on it.
"""

from . import (clasp, closed_forms, compact, consulted, consulted_tree, lm_head, pipeline,  # noqa: F401
               pipeline_async, verify)
