"""Pins of the oracle's gate selection and of the whole-cache oracle."""
import itertools
import math

import numpy as np

from oracle import OracleCache, gate
from workload import WORKLOADS, gen_append_kv, gen_kv, gen_q


def test_d_star_solves_the_meter_equation():
    for tau in (0.0, 0.01, 0.5, 1.0, 2.0, 10.0):
        ds = gate.d_star(tau)
        t32 = float(np.float32(tau))
        assert abs(ds + ds * ds / 2 - t32) < 1e-12 * max(1, t32)


def exceeds(values, ds):
    """Exact sign test of sum(values) - ds > 0 by Shewchuk's exactly rounded sum (math.fsum):
    its result is zero only when the exact sum is, and otherwise has the exact sum's sign."""
    return math.fsum([float(v) for v in values] + [-ds]) > 0.0


def test_selection_is_a_minimum_cardinality_repair_by_brute_force():
    """Over every subset of 9 blocks: the smallest set whose removal leaves remaining risk <= D*
    has exactly as many blocks as the gate's ranked prefix, and the prefix achieves it."""
    rng = np.random.default_rng(0)
    for trial in range(60):
        n = 9
        risk = (rng.exponential(0.05, n) * (rng.random(n) < 0.8)).astype(np.float32)
        rep = rng.random(n) < 0.2
        risk[rep] = 0.0
        tau = float(rng.choice([0.02, 0.05, 0.1, 0.3]))
        ds = gate.d_star(tau)
        sel = gate.select_cell(risk, rep, tau)
        cand = [b for b in range(n) if not rep[b]]
        if not exceeds(risk[cand], ds):
            assert sel == []
            continue
        best = None
        for k in range(len(cand) + 1):
            for sub in itertools.combinations(cand, k):
                if not exceeds([risk[b] for b in cand if b not in sub], ds):
                    best = k
                    break
            if best is not None:
                break
        assert len(sel) == best
        assert not exceeds([risk[b] for b in cand if b not in sel], ds)
        assert not any(rep[b] for b in sel)


def test_selection_ranks_by_risk_then_lower_index():
    risk = np.array([0.1, 0.3, 0.3, 0.05, 0.3], np.float32)
    sel = gate.select_cell(risk, np.zeros(5, bool), tau=gate.d_star(0) + 0.0)   # tau = 0 -> all positive
    assert sel == [1, 2, 4, 0, 3]
    # D* between: stop as soon as the remaining risk fits
    tau = 0.16 + 0.16 ** 2 / 2
    assert gate.select_cell(risk, np.zeros(5, bool), tau) == [1, 2, 4]


def test_group_union_and_persistence():
    risk = np.array([[0.5, 0.0, 0.0, 0.0], [0.0, 0.0, 0.6, 0.0]], np.float32)
    rep = np.array([False, False, False, False])
    assert gate.gate_group(risk, rep, 0.1) == [0, 2]
    rep[0] = True
    assert gate.gate_group(risk, rep, 0.1) == [2]


def test_oracle_cache_gate_lowers_the_meter_next_step():
    """Raw-cast FP8 on the tiny case: after repairing what the gate asks for at tau, the same
    query's meter on the repaired cache is <= tau up to the logit shift the repair itself causes."""
    w = WORKLOADS["tiny"].with_(scheme="fp8_e4m3")
    c = OracleCache(1, w.n_q_heads, w.n_kv_heads, 1, "fp8_e4m3", 0, w.steps)
    K, V = gen_kv(w, 0)
    c.write(0, K, V)
    q = gen_q(w, 0, 0)
    r0 = c.decode(0, q, w.delta_req)
    tau = 0.05
    picked = c.gate(0, tau, r0["risk"].astype(np.float32))
    assert picked, "fp8 raw cast should trigger the gate at tau=0.05"
    r1 = c.decode(0, q, w.delta_req)
    assert np.all(r1["raw_a"] <= np.maximum(r0["raw_a"], 0) + 1e-12)
    assert np.max(r1["raw_a"]) < np.max(r0["raw_a"])
    # zeroed witnesses and zero risk on repaired blocks
    for (i, h, b) in picked:
        assert np.all(c.group_view(0, i, h)[2][b * 16:(b + 1) * 16] == 0)
    g = w.group
    for (i, h, b) in picked:
        assert np.all(r1["risk"][i, h * g:(h + 1) * g, b] == 0)


def test_oracle_cache_append_and_kivi_tail():
    w = WORKLOADS["tiny"].with_(scheme="kivi2", context=40)
    c = OracleCache(1, w.n_q_heads, w.n_kv_heads, 1, "kivi2", 0, w.steps)
    K, V = gen_kv(w, 0)
    c.write(0, K, V)                           # 40 tokens: blocks 0, 1 closed, 8-token tail exact
    assert c.length(0) == 40
    kh, _, wst, _, _ = c.group_view(0, 0, 0)
    np.testing.assert_array_equal(kh[32:], K[0, 32:, 0])
    assert np.all(wst[32:] == 0) and np.any(wst[:32] > 0)
    for step in range(8):
        k1, v1 = gen_append_kv(w, 0, step)
        c.write(0, k1, v1)
    kh, _, wst, _, _ = c.group_view(0, 0, 0)   # 48 tokens: block 2 closed on the last append
    assert np.any(wst[32:48] > 0) and not np.array_equal(kh[32:48], K[0, 32:48, 0])


def test_selection_over_many_blocks_is_the_exact_minimum_repair():
    """Hundreds of blocks: the ranked prefix is the smallest whose exact remaining risk
    (math.fsum sign test) is <= D*; ranking by size makes a prefix the optimum."""
    rng = np.random.default_rng(6)
    for trial in range(40):
        n = int(rng.integers(40, 400))
        risk = (rng.exponential(0.01, n) * (rng.random(n) < 0.9)).astype(np.float32)
        rep = rng.random(n) < 0.1
        total = math.fsum(float(x) for x in risk[~rep])
        tau = float(np.float32(float(rng.uniform(0.05, 0.9)) * (total + total * total / 2)))
        ds = gate.d_star(tau)
        sel = gate.select_cell(risk, rep, tau)
        order = sorted((b for b in range(n) if not rep[b]), key=lambda b: (-float(risk[b]), b))
        k_exact = 0
        while exceeds([risk[b] for b in order[k_exact:]], ds):
            k_exact += 1
        assert sel == order[:k_exact]


def test_exact_ties_and_sums_that_float64_gets_wrong():
    """tau = 1.5 gives D* = 1 exactly and tau = 4 gives D* = 2 (float32 and float64 exact)."""
    assert gate.d_star(1.5) == 1.0 and gate.d_star(4.0) == 2.0
    no = np.zeros(8, bool)
    # the total equals D*: the cell does not trigger; one unit more and it does
    assert gate.select_cell(np.array([0.5, 0.25, 0.25], np.float32), no[:3], 1.5) == []
    tiny = np.float32(2.0 ** -149)
    assert gate.select_cell(np.array([0.5, 0.25, 0.25, tiny], np.float32), no[:4], 1.5) == [0]
    # remaining after the first block is exactly D*: the prefix stops there
    assert gate.select_cell(np.array([0.75, 0.5, 0.5], np.float32), no[:3], 1.5) == [0]
    # 1 + 4 * 2^-60 > 1 although a float64 running sum from the left rounds it to 1
    r = np.array([1.0] + [2.0 ** -60] * 4, np.float32)
    assert sum(float(x) for x in r) == 1.0                # the float64 running sum
    assert gate.select_cell(r, no[:5], 1.5) == [0]
    # equal risks: lower block index first; exactly D* = 2 left after three of five
    r = np.array([0.5, 0.5, 1.0, 0.5, 1.0], np.float32)
    assert gate.select_cell(r, no[:5], 4.0) == [2, 4]
    assert gate.select_cell(r, no[:5], 1.5) == [2, 4, 0]


def test_tau_zero_takes_every_positive_risk():
    r = np.array([0.0, 1e-30, 0.0, 3.0, 2.0 ** -149], np.float32)
    assert gate.d_star(0.0) == 0.0
    assert gate.select_cell(r, np.zeros(5, bool), 0.0) == [3, 1, 4]


def test_nan_counts_as_infinite_and_negative_as_zero():
    r = np.array([0.1, np.nan, np.inf, -1.0, 0.2], np.float32)
    # NaN and +inf are taken first (ties to the lower index), then by size until <= D*
    assert gate.select_cell(r, np.zeros(5, bool), 0.05) == [1, 2, 4, 0]
    assert gate.select_cell(r, np.zeros(5, bool), 10.0) == [1, 2]
    assert gate.select_cell(np.array([-1.0, -0.0], np.float32), np.zeros(2, bool), 0.0) == []


def test_tau_is_read_as_float32():
    """The library's gate takes tau as a float: 0.2 means float32(0.2), not the double 0.2."""
    assert gate.d_star(0.2) == math.sqrt(1.0 + 2.0 * float(np.float32(0.2))) - 1.0
    assert gate.d_star(0.2) != math.sqrt(1.0 + 2.0 * 0.2) - 1.0
