"""CPU oracle for the metered KV-cache decode path — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 numpy statement of what the path computes: the dither
stream, the three cache writers and the band-norm witness, the Tier A bound,
the Tier B certificate, the total-variation meter, split-KV partial states and
their log-sum-exp merge, and the gate's block selection.  It shares no code,
tables or constants with the CUDA library and neither imports the other; only
the seeded input generators in `workload/` serve both.

Only `tests/`, `__graft_entry__.smoke()` and the `cpu_baseline` / reference leg
of `bench.py` may import or run anything in this package.  The product path
never falls back to it.

Citations name the pages the method is taken from, all titled
"WitCert: Sound Runtime Risk Observability and Gating for KV-Cache
Quantization":
  [WitCert summary]   the technical summary page (montaan.com): witness
                      paragraph with Lemma 1, Theorem 2, the Tier B paragraph,
                      the implementation paragraph, the results paragraphs and
                      the closing list of improvements (TV bound formula);
  [WitCert abstract]  the arXiv abstract (mlsanity.com index page);
  [WitCert Lean page] the paperswithlean.com page: Approach, Figure 2 and
                      Figure 5 captions.
Philox4x32-10 follows Salmon et al., "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11).

Parity pins: every function here is pinned by a `-m "not gpu"` test against
published vectors, closed forms, invariants or brute force (tests/test_oracle_*.py).
"""
from . import fp, gate, meter, philox, quant  # noqa: F401
from .cache import OracleCache  # noqa: F401
