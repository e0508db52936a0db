"""The gate's block selection on the GPU (witcert_gate_select) against the oracle's rule.

The oracle ranks a cell's unrepaired blocks and takes the shortest prefix whose exact
remaining risk is <= D*(tau); the GPU must pick exactly the same blocks, bit for bit, including
where plain floating-point sums would decide otherwise: totals exactly equal to D*, remaining
sums that hit D* exactly, sums that float64 rounds to D*, equal risks (lower block first), NaN
and infinite risks, tau = 0.  Block counts cover every sort width the kernel has (up to 16384
blocks per cell).
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from oracle.gate import gate_group

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


def gpu_select(risk, n_kv_heads, tau, repaired=None):
    """Selected blocks per (sequence, KV head) as boolean [B, Hkv, nblk]."""
    B, Hq, nblk = risk.shape
    r = torch.from_numpy(np.ascontiguousarray(risk, np.float32)).cuda()
    rep = None if repaired is None else torch.from_numpy(np.ascontiguousarray(repaired, np.uint8)).cuda()
    words = wc.witcert_gate_select(r, n_kv_heads, tau, rep).cpu().numpy().view(np.uint32)
    bits = (words[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(B, n_kv_heads, -1)[..., :nblk].astype(bool)


def oracle_select(risk, n_kv_heads, tau, repaired=None):
    B, Hq, nblk = risk.shape
    g = Hq // n_kv_heads
    rep = np.zeros((B, n_kv_heads, nblk), bool) if repaired is None else np.asarray(repaired, bool)
    out = np.zeros((B, n_kv_heads, nblk), bool)
    for i in range(B):
        for h in range(n_kv_heads):
            out[i, h, gate_group(risk[i, h * g:(h + 1) * g], rep[i, h], tau)] = True
    return out


def one_cell(values):
    return np.asarray(values, np.float32)[None, None, :]


CRAFTED = [
    ([0.5, 0.25, 0.25], 1.5),                        # total == D* = 1: no trigger
    ([0.5, 0.25, 0.25, 2.0 ** -149], 1.5),           # one unit above: triggers, takes block 0
    ([0.75, 0.5, 0.5], 1.5),                         # remaining exactly D* after one block
    ([1.0] + [2.0 ** -60] * 4, 1.5),                 # float64 running sum says 1 == D*
    ([0.5, 0.5, 1.0, 0.5, 1.0], 4.0),                # equal risks: lower index first
    ([0.5, 0.5, 1.0, 0.5, 1.0], 1.5),
    ([0.0, 1e-30, 0.0, 3.0, 2.0 ** -149], 0.0),      # tau = 0 takes every positive risk
    ([0.1, np.nan, np.inf, -1.0, 0.2], 0.05),        # NaN and inf first, negative is zero
    ([0.1, np.nan, np.inf, -1.0, 0.2], 10.0),
    ([-1.0, -0.0], 0.0),
    ([3.0e38, 3.0e38, 3.0e38], 1e30),                # sums beyond float32's range
]


@pytest.mark.parametrize("values,tau", CRAFTED)
def test_crafted_ties_match_the_exact_rule(values, tau):
    r = one_cell(values)
    np.testing.assert_array_equal(gpu_select(r, 1, tau), oracle_select(r, 1, tau))


@pytest.mark.parametrize("nblk", [1, 37, 511, 512, 513, 1500, 2049, 4100, 9000, 16384])
def test_random_dyadic_risks_with_exact_ties(nblk):
    """Risks on a coarse dyadic grid (many equal values, sums that hit D* exactly) and on a
    continuous scale, some blocks repaired, thresholds whose D* is dyadic (0.25, 0.5, 1) and
    others; query-head groups of 4 on 2 KV heads and 2 sequences."""
    rng = np.random.default_rng(nblk)
    B, Hkv, g = 2, 2, 4
    grid = rng.integers(0, 9, size=(B, Hkv * g, nblk)).astype(np.float32) * np.float32(2.0 ** -10)
    cont = (rng.exponential(1.0, (B, Hkv * g, nblk)) * 10.0 ** rng.uniform(-30, -1, (B, Hkv * g, nblk)))
    risk = np.where(rng.random((B, Hkv * g, nblk)) < 0.5, grid, cont.astype(np.float32)).astype(np.float32)
    risk[rng.random(risk.shape) < 0.05] = 0.0
    repaired = rng.random((B, Hkv, nblk)) < 0.2
    for tau in (0.28125, 0.625, 1.5, 0.0, 0.013, 3.7):
        np.testing.assert_array_equal(gpu_select(risk, Hkv, tau, repaired), oracle_select(risk, Hkv, tau, repaired),
                                      err_msg=f"tau {tau}")


def test_selection_rejects_bad_shapes():
    r = torch.zeros((1, 4, 16385), dtype=torch.float32, device="cuda")
    with pytest.raises(wc.WitcertError) as e:
        wc.witcert_gate_select(r, 1, 1.0)
    assert e.value.status == _lib.EINVAL
    with pytest.raises(wc.WitcertError) as e:
        wc.witcert_gate_select(torch.zeros((1, 3, 16), dtype=torch.float32, device="cuda"), 2, 1.0)
    assert e.value.status == _lib.EINVAL
