"""CPU fp64 oracle for batched Gram Newton-Schulz and the Muon step around it.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links this
package: only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
use it. It shares no code with the CUDA library; its only common dependency is the
seeded input generator (``matrix_orthogonalizing_optimizer_gb300.inputs``), which the
tests call to make the arrays handed to both sides.

Every function is a plain restatement of the pages' definitions and algorithms, in
float64, with numpy's matmul / SVD / sort as library steps and no blocking, fusion or
reordering beyond what the algorithm states:

* ``newton_schulz``: standard Newton-Schulz (Dion3 Algorithm 1), naive Gram
  Newton-Schulz (Dion3 Algorithm 2), stabilized Gram Newton-Schulz with restart
  (Dion3 Algorithm 3), the scalar recurrence of Dion3 Theorem 2 and the
  composition of the odd polynomials, polar(X) from the SVD (Dion3 Definition 1),
  and the FLOP accounting of Dion3 sections 2.2, 2.3, 4.1 and 4.2.
* ``muon``: the Muon step (Dion3 eq. (1)), the Dion3 fractional update (Dion3
  Algorithm 4 and section 6), exact l1 row keys and top-k selection.
* ``stability``: the spectrum experiments of Dion3 appendix B (eigenvalue tracking with
  the diagonalisation error, restart-location sweep).

Parity unpinned: none of the functions above; every one is pinned in
``tests/test_oracle_pins.py`` against closed forms, SVD, brute force or the pages'
printed numbers (``stability.spectrum_trace`` against the polynomial composition in the
singular basis, ``stability.restart_sweep`` against the matrix form of Algorithm 3 with the
planted eigenvalue). What stays unpinned is outside the oracle: training quality
(validation perplexity) and the Polar Express coefficient values, which no page prints.
"""
from . import newton_schulz, muon, stability  # noqa: F401
