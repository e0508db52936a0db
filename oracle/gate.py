"""Meter-driven gate of the oracle: which exact key blocks to page in.

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

D and the remaining risks are suffix sums of the ranked risks in float64; the
risks themselves are the fp32 values the decode reported.  Repaired blocks
carry zero risk and are not ranked.  The pages fix no summation order; this
reading fixes one so that the choice is reproducible bit for bit: the ranked
list is cut into runs of RUN consecutive blocks, each run is summed from its
lowest-ranked block upward, the run totals are summed from the last run
upward, and the remaining risk after block j is (j's run-local suffix) + (the
total of the runs after j's run).
"""
from __future__ import annotations

import math

import numpy as np


def d_star(tau: float) -> float:
    """Solution of D + D^2/2 = tau."""
    return math.sqrt(1.0 + 2.0 * tau) - 1.0


RUN = 32


def suffix_sums(values):
    """Remaining-risk sums of a ranked list: entry k = sum of values[k:], in the run order above;
    entry len(values) = 0."""
    n = len(values)
    local = [0.0] * n
    totals = []
    for lo in range(0, n, RUN):
        s = 0.0
        for k in range(min(n, lo + RUN) - 1, lo - 1, -1):
            s = s + float(values[k])
            local[k] = s
        totals.append(s)
    after = [0.0] * len(totals)          # total of the runs after run c
    u = 0.0
    for c in range(len(totals) - 1, -1, -1):
        after[c] = u
        u = u + totals[c]
    return [local[k] + after[k // RUN] for k in range(n)] + [0.0]


def select_cell(risk_row, repaired, tau: float):
    """Blocks one (sequence, query head) cell asks for.  risk_row: fp32 [nblk]."""
    r = np.asarray(risk_row, dtype=np.float32)
    cand = np.nonzero(~np.asarray(repaired, bool))[0]
    if cand.size == 0:
        return []
    # rank: larger risk first, ties to the lower block index
    order = sorted(cand.tolist(), key=lambda b: (-float(r[b]), b))
    suffix = suffix_sums([r[b] for b in order])
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
