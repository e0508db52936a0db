"""Host-side helpers of bench.py (no GPU): the kernel-source digest that keys recorded
profile counters, the ragged-context draw and the per-token byte accounting."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_kernel_digest_ignores_comments_but_not_code(bench, tmp_path):
    a = tmp_path / "a.cuh"
    a.write_text("// header\nint f(int x) {\n  return x + 1;   // one more\n}\n")
    b = tmp_path / "b.cuh"
    b.write_text("int f(int x) {\n\n  return x + 1;\n}\n// trailing note\n")
    c = tmp_path / "c.cuh"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.kernel_digest(a) == bench.kernel_digest(b)
    assert bench.kernel_digest(a) != bench.kernel_digest(c)
    assert len(bench.kernel_digest(a)) == 16


def test_ragged_lengths_are_seeded_and_in_range(bench):
    from workload import WORKLOADS
    w = WORKLOADS["qwen_28l"]
    lens = bench.ragged_lengths(w, "512:4096")
    assert lens == bench.ragged_lengths(w, "512:4096")
    assert len(lens) == w.batch and all(512 <= n <= 4096 for n in lens) and len(set(lens)) > 1
    assert bench.ragged_lengths(w, None) == [w.context] * w.batch
    with pytest.raises(AssertionError):
        bench.ragged_lengths(w, "512:99999")


def test_bytes_per_token_head_match_the_oracle_accounting(bench):
    from oracle import quant
    assert bench.BYTES_PER_TOK_HEAD == quant.BYTES_PER_TOKEN_HEAD
    assert bench.tok_head_bytes("int8_dither", True) == 304 + quant.V_WITNESS_BYTES


def test_timed_launch_count_follows_the_write_path(bench):
    """Three launches per layer and step on the default path (writer, split, merge); KIVI adds
    its key writer; a ragged cache adds the length push; a paged cache adds one page-table push
    in each step where a sequence starts a block."""
    t = bench.timed_launches
    assert t("int8_dither", 28, [4096] * 16, 10, False, False) == 3 * 28 * 10
    assert t("fp8_e4m3", 28, [4096] * 16, 10, False, False) == 3 * 28 * 10
    assert t("kivi2", 28, [4096] * 16, 10, False, False) == 4 * 28 * 10
    assert t("int8_dither", 28, [600, 4000], 10, True, False) == 4 * 28 * 10
    assert t("kivi2", 2, [600, 4000], 10, True, False) == (4 + 2) * 2 * 10
    # one sequence at 4096 starts a block at steps 0 and 16; two at 4100 both start one at
    # step 12, which takes one push
    assert t("int8_dither", 1, [4096], 20, False, True) == 3 * 20 + 2
    assert t("int8_dither", 1, [4100, 4100], 20, True, True) == 4 * 20 + 1


def test_l2_note_says_when_a_cache_can_stay_in_l2(bench):
    """Below twice L2 the bench line says the steps may hit L2; above it that they read HBM."""
    assert bench.l2_note(40e6).startswith("cache of 0.040 GB within twice L2")
    assert bench.l2_note(2 * bench.L2_BYTES + 1).startswith("inputs larger than L2")
    from workload import sweep_workload
    w = sweep_workload("mistral", 16, 32768)
    assert w.batch * w.n_kv_heads * w.context * 304 * 32 > 2 * bench.L2_BYTES     # the default line
