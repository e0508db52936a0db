"""Meter-driven gate of the oracle: which exact key blocks to page in.

Per the pages, once the meter passes a threshold the gate brings exact keys
back from host memory a block at a time and clears the witnesses of what it
repaired; it ranks by risk when the threshold is 1 or more and certifies below
1, and repairs accumulate and persist
[WitCert summary, implementation paragraph; WitCert Lean page, Approach and
Figures 2 and 5].  The ranking and stopping rule below are this build's
reading of those sentences:

* a (sequence, query head) cell triggers when its unclamped meter
  D + D^2/2 exceeds tau, i.e. when D > D*(tau) = sqrt(1 + 2 tau) - 1;
* its unrepaired blocks are ranked by risk R_blk (share of D), largest first,
  ties to the lower block index;
* it takes the shortest prefix after which the remaining risk is <= D*(tau),
  which brings the cell's meter to <= tau from the next step on;
* a block is repaired once any query head of its KV head's group selects it.

D and the remaining risks are suffix sums of the ranked risks, accumulated in
float64 from the lowest-ranked block upward; the risks themselves are the fp32
values the decode reported.  Repaired blocks carry zero risk and are not ranked.
"""
from __future__ import annotations

import math

import numpy as np


def d_star(tau: float) -> float:
    """Solution of D + D^2/2 = tau."""
    return math.sqrt(1.0 + 2.0 * tau) - 1.0


def select_cell(risk_row, repaired, tau: float):
    """Blocks one (sequence, query head) cell asks for.  risk_row: fp32 [nblk]."""
    r = np.asarray(risk_row, dtype=np.float32)
    cand = np.nonzero(~np.asarray(repaired, bool))[0]
    if cand.size == 0:
        return []
    # rank: larger risk first, ties to the lower block index
    order = sorted(cand.tolist(), key=lambda b: (-float(r[b]), b))
    n = len(order)
    suffix = [0.0] * (n + 1)
    for k in range(n - 1, -1, -1):
        suffix[k] = suffix[k + 1] + float(r[order[k]])
    ds = d_star(tau)
    if not suffix[0] > ds:
        return []
    k = 0
    while suffix[k] > ds:
        k += 1
    return order[:k]


def gate_group(risk, repaired, tau: float):
    """Union over the query heads of one KV head's group.  risk: [g, nblk]."""
    sel = set()
    for j in range(risk.shape[0]):
        sel.update(select_cell(risk[j], repaired, tau))
    return sorted(sel)
