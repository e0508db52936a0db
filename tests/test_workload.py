"""The seeded generators: determinism, dtype exactness, and the structure they promise."""
import math

import numpy as np

from workload import (WORKLOADS, bf16_bits, bf16_from_bits, bf16_round, gen_append_kv, gen_kv,
                      gen_q, planted_positions, sweep_workload)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    got = bf16_round(x)
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == -2.5
    np.testing.assert_array_equal(bf16_from_bits(bf16_bits(got)), got)


def test_generators_are_deterministic_and_exact_in_dtype():
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=64)
    K1, V1 = gen_kv(w, 0)
    K2, V2 = gen_kv(w, 0)
    np.testing.assert_array_equal(K1, K2)
    np.testing.assert_array_equal(bf16_round(K1), K1)
    assert K1.shape == (2, 64, 4, 128)
    q = gen_q(w, 0, 3)
    assert q.shape == (2, 28, 128)
    np.testing.assert_array_equal(bf16_round(q), q)
    assert not np.array_equal(gen_q(w, 0, 4), q)
    k1, v1 = gen_append_kv(w, 0, 0)
    assert k1.shape == (2, 1, 4, 128)


def test_planted_key_scores_about_eight():
    w = WORKLOADS["qwen_1l"].with_(batch=4, context=512)
    K, _ = gen_kv(w, 0)
    q = gen_q(w, 0, 0)
    pos = planted_positions(w, 0)
    for i in range(w.batch):
        logit = q[i, 0] @ K[i, pos[i], 0] / math.sqrt(128)
        assert 6.0 < logit < 10.0


def test_outliers_sit_on_one_rope_pair():
    w = WORKLOADS["qwen_1l"].with_(batch=1, context=2048, planted=False)
    K, _ = gen_kv(w, 0)
    e = (K[0, :, 0].astype(np.float64) ** 2).mean(0)
    assert e[10] + e[74] > 0.9 * e.sum()
    assert abs(e[10] - e[74]) < 0.2 * e[10]       # rotation spreads the pair's energy evenly


def test_sweep_shapes():
    m = sweep_workload("mistral", 4, 8192)
    y = sweep_workload("yi", 1, 131072, "fp8_e4m3")
    assert (m.n_q_heads, m.n_kv_heads, m.rope_base) == (32, 8, 1e4)
    assert (y.n_q_heads, y.n_kv_heads, y.rope_base, y.scheme) == (32, 4, 5e6, "fp8_e4m3")
