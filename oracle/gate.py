"""Meter-driven gate of the oracle: which exact key blocks to page in.

Test infrastructure: a plain statement of the gate's selection rule, used by the tests,
the smoke check and the benchmark's CPU baseline only, never by the library.

Per the pages, once the meter passes a threshold the gate brings exact keys
back from host memory a block at a time and clears the witnesses of what it
repaired; it ranks by risk when the threshold is 1 or more and certifies below
1, and repairs accumulate and persist
[WitCert summary, implementation paragraph; WitCert Lean page, Approach and
Figures 2 and 5].  The ranking and stopping rule below are a reading of
those sentences (the pages state the behavior, not the rule):

* a (sequence, query head) cell triggers when its unclamped meter
  D + D^2/2 exceeds tau, i.e. when D > D*(tau) = sqrt(1 + 2 tau) - 1;
* its unrepaired blocks are ranked by risk R_blk (share of D), largest first,
  ties to the lower block index;
* it takes the shortest prefix after which the remaining risk is <= D*(tau),
  which brings the cell's meter to <= tau from the next step on;
* a block is repaired once any query head of its KV head's group selects it.

D and the remaining risks are the exact sums of the fp32 risks the decode
reported (exact rationals: no summation order, no rounding), compared exactly
with D*(tau) evaluated in float64 from tau as a float32 (the library's gate
takes tau as a float).  Repaired blocks are not ranked.  A risk that is not a
number counts as +infinity (such a block is always taken, first); a risk that
is not positive counts as zero.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def d_star(tau) -> float:
    """Solution of D + D^2/2 = tau, in float64, for tau rounded to float32."""
    return math.sqrt(1.0 + 2.0 * float(np.float32(tau))) - 1.0


def canonical_risk(r) -> float:
    """The fp32 risk as the rule reads it: NaN -> +inf, anything not positive -> 0."""
    x = float(np.float32(r))
    if math.isnan(x):
        return math.inf
    return x if x > 0.0 else 0.0


def select_cell(risk_row, repaired, tau):
    """Blocks one (sequence, query head) cell asks for.  risk_row: fp32 [nblk]."""
    rep = np.asarray(repaired, bool)
    r = [canonical_risk(x) for x in np.asarray(risk_row, dtype=np.float32)]
    cand = [b for b in range(len(r)) if not rep[b]]
    if not cand:
        return []
    # rank: larger risk first, ties to the lower block index
    order = sorted(cand, key=lambda b: (-r[b], b))
    n_inf = sum(1 for b in cand if r[b] == math.inf)
    remaining = sum((Fraction(r[b]) for b in cand if r[b] != math.inf), Fraction(0))
    ds = Fraction(d_star(tau))
    if n_inf == 0 and not remaining > ds:
        return []
    k = n_inf                     # infinite risks come first and are always taken
    while remaining > ds:
        remaining -= Fraction(r[order[k]])
        k += 1
    return order[:k]


def gate_group(risk, repaired, tau):
    """Union over the query heads of one KV head's group.  risk: [g, nblk]."""
    sel = set()
    for j in range(risk.shape[0]):
        sel.update(select_cell(risk[j], repaired, tau))
    return sorted(sel)
