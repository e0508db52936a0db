"""Pins of the oracle's gate selection and of the whole-cache oracle."""
import itertools
import math

import numpy as np

from oracle import OracleCache, gate
from workload import WORKLOADS, gen_append_kv, gen_kv, gen_q


def test_d_star_solves_the_meter_equation():
    for tau in (0.0, 0.01, 0.5, 1.0, 2.0, 10.0):
        ds = gate.d_star(tau)
        assert abs(ds + ds * ds / 2 - tau) < 1e-12 * max(1, tau)


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
        total = float(np.sum(risk.astype(np.float64)))
        if not total > ds:
            assert sel == []
            continue
        cand = [b for b in range(n) if not rep[b]]
        best = None
        for k in range(len(cand) + 1):
            for sub in itertools.combinations(cand, k):
                rest = total - sum(float(risk[b]) for b in sub)
                if rest <= ds + 1e-12:
                    best = k
                    break
            if best is not None:
                break
        assert len(sel) == best
        assert total - sum(float(risk[b]) for b in sel) <= ds + 1e-12
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


def test_run_order_suffix_sums_match_exact_sums_and_are_monotone():
    """The fixed summation order stays within float64 rounding of the exact remaining risk
    (math.fsum) and never increases down the ranked list, over several runs of 32."""
    rng = np.random.default_rng(5)
    for n in (1, 31, 32, 33, 100, 257, 2048):
        vals = np.sort((rng.exponential(1.0, n) ** 4 * 10.0 ** rng.uniform(-12, 0, n)).astype(np.float32))[::-1]
        suf = gate.suffix_sums(vals)
        assert len(suf) == n + 1 and suf[n] == 0.0
        for k in range(0, n, max(1, n // 50)):
            exact = math.fsum(float(v) for v in vals[k:])
            assert abs(suf[k] - exact) <= 1e-13 * exact
        assert all(suf[k] >= suf[k + 1] for k in range(n))


def test_selection_over_many_runs_is_the_exact_minimum_repair():
    """Hundreds of blocks (many runs): the ranked prefix is the smallest whose exact remaining
    risk (math.fsum) is <= D*; ranking by size makes a prefix the optimum."""
    rng = np.random.default_rng(6)
    for trial in range(40):
        n = int(rng.integers(40, 400))
        risk = (rng.exponential(0.01, n) * (rng.random(n) < 0.9)).astype(np.float32)
        rep = rng.random(n) < 0.1
        risk[rep] = 0.0
        total = math.fsum(float(x) for x in risk)
        tau = float(rng.uniform(0.05, 0.9)) * (total + total * total / 2)
        ds = gate.d_star(tau)
        sel = gate.select_cell(risk, rep, tau)
        order = sorted((b for b in range(n) if not rep[b]), key=lambda b: (-float(risk[b]), b))
        k_exact = 0
        while math.fsum(float(risk[b]) for b in order[k_exact:]) > ds:
            k_exact += 1
        assert sel == order[:k_exact]
