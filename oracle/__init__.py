"""Float64 CPU oracle for the log-space dense sum layer and the circuits built on it.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product (``log_space_sum_gb300``) never imports it, and this
package never imports the product: the two share no code. The only module both
sides use is ``workloads`` (seeded input draws, none of the method's arithmetic).

Everything here is plain NumPy in float64, written for a reader to check against
the pages by eye:

* ``sum_layer`` - the dense sum layer forward (log-space) and its EM flows
  (pyjuice PR #62, Summary 2 and 3).
* ``hmm``       - the HMM circuit as a chain of shared-children sum layers
  (pyjuice PR #62, Summary 2, first bullet; Results table).
* ``hclt``      - the HCLT circuit as a tree of per-edge sum layers
  (pyjuice PR #62, Summary 2, second bullet; Results table).
* ``lowrank``   - the LowRank ``exp_sum`` per-sample scale and its backward
  statistics (pyjuice LowRank API doc: intro formulas, Training).
* ``emulate``   - a precision emulator (bf16 RNE, TF32 round-to-nearest, 3xTF32
  splits) used only to predict the error envelope of each precision mode
  (pyjuice PR #62, Summary 1 table). It is not a pin of correctness.

Every function is pinned in ``tests/test_oracle_*.py`` by closed forms, brute
force enumeration, invariants and finite differences.
"""
from . import sum_layer, hmm, hclt, lowrank, emulate  # noqa: F401
