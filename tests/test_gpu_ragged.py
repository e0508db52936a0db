"""Ragged batches on the GPU: sequences of different lengths in one cache, in a contiguous
store and in a paged one (a shared pool of pages behind a per-sequence page table).

Each sequence of the GPU cache is checked against its own single-sequence oracle
cache (the oracle of one sequence is the plain definition: its tokens, its
positions, its length as S in Tier B).  Covers a ragged prefill (an empty
sequence, a ragged tail, lengths spanning several splits), ragged appends with
some sequences idle, a sequence reset and refill (continuous batching), the gate
on ragged lengths, and every scheme with value witnesses on; the paged store must
give the same results with a pool far smaller than batch x max_tokens.
"""
import numpy as np
import pytest
import torch

import kv_cache_quantization_witcert_gb300 as wc
from kv_cache_quantization_witcert_gb300 import _lib
from oracle import OracleCache
from workload import WORKLOADS, gen_kv, gen_q

from gpu_helpers import METER_REL, check_gate_end_to_end, check_meter, check_risk, tensor_function, torch_dtype

pytestmark = pytest.mark.gpu

ALL_SCHEMES = ["int8_dither", "fp8_e4m3", "kivi2", "int8_rtn", "blackbox"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    wc.load()


class Ragged:
    """A GPU cache of B sequences and one oracle cache per sequence."""

    def __init__(self, w, scheme, cap, v_witness=True, gate_blocks=0, n_splits=0, max_pages=0):
        self.w, self.scheme, self.B = w, scheme, w.batch
        self.gpu = wc.Cache(w.n_layers, w.n_q_heads, w.n_kv_heads, w.batch, cap, scheme, dtype=torch_dtype(w),
                            seed=w.seed, total_steps=w.steps, max_repair_blocks=gate_blocks, v_witness=v_witness,
                            n_splits=n_splits, max_pages=max_pages)
        self.refs = [OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, 1, scheme, w.seed, w.steps,
                                 v_witness=v_witness) for _ in range(w.batch)]
        self.fseed = 0

    def dev(self, x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device="cuda").to(torch_dtype(self.w))

    def write(self, layer, parts):
        """parts[i]: (K_i, V_i) of shape [n_i, Hkv, d] (n_i may be 0)."""
        counts = [p[0].shape[0] for p in parts]
        K = np.concatenate([p[0] for p in parts], 0)
        V = np.concatenate([p[1] for p in parts], 0)
        Kd, Vd = self.dev(K), self.dev(V)
        if self.scheme == "blackbox":
            self.fseed += 2
            Kh, Vh = self.dev(tensor_function(K, self.fseed)), self.dev(tensor_function(V, self.fseed + 1))
            self.gpu.witcert_write_ragged(layer, Kd, Vd, counts, Kh, Vh)
            Kh, Vh = Kh.float().cpu().numpy(), Vh.float().cpu().numpy()
        else:
            self.gpu.witcert_write_ragged(layer, Kd, Vd, counts)
        row = 0
        for i, n in enumerate(counts):
            if n:
                sl = slice(row, row + n)
                if self.scheme == "blackbox":
                    self.refs[i].write(layer, K[None, sl], V[None, sl], Kh[None, sl], Vh[None, sl])
                else:
                    self.refs[i].write(layer, K[None, sl], V[None, sl])
            row += n
        for i in range(self.B):
            assert self.gpu.witcert_seq_length(layer, i) == self.refs[i].length(layer)

    def check_store(self, layer):
        """Stored witnesses (and value witnesses) of every sequence's own rows, bit for bit."""
        w16 = self.gpu.export(layer, _lib.X_WITNESS).cpu().numpy()
        wv = self.gpu.export(layer, _lib.X_V_WITNESS).cpu().numpy() if self.gpu.v_witness else None
        for i, ref in enumerate(self.refs):
            S = ref.length(layer)
            np.testing.assert_array_equal(w16[i, :S].view(np.uint16), ref.w16[layer][0].view(np.uint16))
            if wv is not None:
                np.testing.assert_array_equal(wv[i, :S].view(np.uint16), ref.wv16[layer][0].view(np.uint16))

    def check_decode(self, layer, q, delta_req):
        out, m = self.gpu.decode(layer, self.dev(q), delta_req)
        o = out.cpu().numpy()
        mm = {k: v.cpu().numpy() for k, v in m.items()}
        w16 = self.gpu.export(layer, _lib.X_WITNESS).cpu().numpy()
        risks = []
        for i, ref in enumerate(self.refs):
            S = ref.length(layer)
            ref.w16[layer] = w16[i:i + 1, :S]
            r = ref.decode(layer, q[i:i + 1], delta_req)
            vmax = np.abs(ref.v[layer]).max() if S else 1.0
            assert np.abs(o[i] - r["out"][0]).max() <= 2e-3 * vmax, f"sequence {i} (S={S})"
            check_meter(mm["raw_a"][i], r["raw_a"][0], METER_REL, f"raw_a seq {i}", raw=True)
            if self.scheme == "int8_dither":
                check_meter(mm["raw_b"][i], r["raw_b"][0], METER_REL, f"raw_b seq {i}", raw=True)
            if self.gpu.v_witness:
                check_meter(mm["meter_v"][i], r["meter_v"][0], METER_REL, f"meter_v seq {i}")
            if S == 0:
                assert not np.any(o[i]) and mm["raw_a"][i].max() == 0
            risks.append(r["risk"][0])
        return out, mm, risks


def _split(arr, lens, start=None):
    """Per-sequence slices [n_i, Hkv, d] of arr [B, S, Hkv, d], from start[i] (0) on."""
    start = start or [0] * len(lens)
    return [arr[i, start[i]:start[i] + n] for i, n in enumerate(lens)]


@pytest.mark.parametrize("pages", [0, 100])
@pytest.mark.parametrize("scheme", ALL_SCHEMES)
def test_ragged_prefill_appends_and_reset(scheme, pages):
    """Four sequences of lengths 0 / 37 / 300 / 1000 (an empty one, ragged tails, several
    splits), then appends of 1 / 0 / 3 / 1 tokens, then sequence 2 reset and refilled; with a
    contiguous store and with a pool of 100 pages (4 x 1100 tokens would take 276)."""
    w = WORKLOADS["qwen_1l"].with_(batch=4, context=1000, steps=3, scheme=scheme)
    rg = Ragged(w, scheme, cap=1100, max_pages=pages)
    K, V = gen_kv(w, 0)
    lens = [0, 37, 300, 1000]
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    rg.check_store(0)
    rg.check_decode(0, gen_q(w, 0, 0), w.delta_req)
    K2, V2 = gen_kv(w.with_(context=16), 5)
    app = [1, 0, 3, 1]
    rg.write(0, list(zip(_split(K2, app), _split(V2, app))))
    rg.check_store(0)
    rg.check_decode(0, gen_q(w, 0, 1), w.delta_req)
    if pages:
        assert rg.gpu.witcert_stats()["pages_used"] == 1 + 3 + 19 + 63
    rg.gpu.witcert_reset_sequence(2)
    rg.refs[2] = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, 1, scheme, w.seed, w.steps, v_witness=True)
    assert rg.gpu.witcert_seq_length(0, 2) == 0
    if pages:
        assert rg.gpu.witcert_stats()["pages_used"] == 1 + 3 + 63
    rg.check_decode(0, gen_q(w, 0, 2), w.delta_req)
    K3, V3 = gen_kv(w.with_(context=64), 6)
    refill = [0, 0, 50, 0]
    rg.write(0, list(zip(_split(K3, refill), _split(V3, refill))))
    rg.check_store(0)
    rg.check_decode(0, gen_q(w, 0, 2), 1e-3)
    assert rg.gpu.witcert_stats()["device_errors"] == 0


def test_ragged_single_token_appends_cross_block_boundaries():
    """Tiny fp32 INT8-dither, three sequences at different offsets inside a block, 20 rounds
    of single-token appends to a changing subset (KIVI-free path of the ragged kernel and the
    dither of each sequence's own positions)."""
    w = WORKLOADS["tiny"].with_(batch=3, context=40, steps=20)
    rg = Ragged(w, "int8_dither", cap=80, n_splits=3)
    K, V = gen_kv(w, 0)
    lens = [5, 16, 29]
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    Ka, Va = gen_kv(w.with_(context=40), 3)
    pos = [0, 0, 0]
    for step in range(20):
        app = [1 if (step + i) % (i + 1) == 0 else 0 for i in range(3)]
        rg.write(0, list(zip(_split(Ka, app, pos), _split(Va, app, pos))))
        pos = [p + a for p, a in zip(pos, app)]
        if step % 5 == 4:
            rg.check_store(0)
            rg.check_decode(0, gen_q(w, 0, step), w.delta_req)


def test_ragged_kivi_appends_close_blocks_per_sequence():
    w = WORKLOADS["tiny"].with_(batch=3, context=40, steps=20, scheme="kivi2")
    rg = Ragged(w, "kivi2", cap=80)
    K, V = gen_kv(w, 0)
    lens = [14, 15, 31]
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    Ka, Va = gen_kv(w.with_(context=40), 3)
    pos = [0, 0, 0]
    for step in range(6):
        app = [2, 1, 3]
        rg.write(0, list(zip(_split(Ka, app, pos), _split(Va, app, pos))))
        pos = [p + a for p, a in zip(pos, app)]
        rg.check_store(0)
        rg.check_decode(0, gen_q(w, 0, step), w.delta_req)


@pytest.mark.parametrize("pages", [0, 60])
@pytest.mark.parametrize("scheme", ["fp8_e4m3", "int8_dither"])
def test_ragged_gate_decisions_match_each_sequence(scheme, pages):
    """FP8 (Tier A risks) and dithered INT8 (Tier B risks) with the gate on ragged lengths: each
    sequence's block risks (its own blocks; the GPU's rows past its length are zero) match its
    oracle's, drive that sequence's oracle gate, and the GPU pages in exactly those blocks
    (witnesses zeroed in the page that holds each block when paged); the oracle's own risks give
    the same blocks outside the tie zone (empty here)."""
    w = WORKLOADS["qwen_1l"].with_(batch=3, context=500, steps=3, scheme=scheme)
    rg = Ragged(w, scheme, cap=520, v_witness=False, gate_blocks=3 * 4 * 40, max_pages=pages)
    K, V = gen_kv(w, 0)
    lens = [500, 130, 257]
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    for step, tau in enumerate((0.5, 0.1) if scheme == "fp8_e4m3" else (4.0, 2.0)):
        _, _, oracle_risk = rg.check_decode(0, gen_q(w, 0, step), w.delta_req)
        risk = rg.gpu.export(0, _lib.X_BLOCK_RISK).cpu().numpy()
        before = [ref.repaired[0][0].copy() for ref in rg.refs]
        rg.gpu.witcert_gate(0, tau)
        slots = rg.gpu.export(0, _lib.X_SLOTS).cpu().numpy()
        for i, ref in enumerate(rg.refs):
            nblk = (lens[i] + 15) // 16
            assert not np.any(risk[i, :, nblk:])
            check_risk(risk[i, :, :nblk], oracle_risk[i], what=f"block risk seq {i}")
            ref.gate(0, tau, risk[i:i + 1, :, :nblk])
            np.testing.assert_array_equal(slots[i, :, :nblk] >= 0, ref.repaired[0][0])
            assert not np.any(slots[i, :, nblk:] >= 0)
            assert check_gate_end_to_end(oracle_risk[i][None], before[i][None], tau, slots[i:i + 1, :, :nblk] >= 0,
                                         w.group) == 0
    rg.check_decode(0, gen_q(w, 0, 7), w.delta_req)
    assert rg.gpu.witcert_gate_stats()["blocks_paged_in"] > 0


def _gate_check(rg, layer, tau, lens, oracle_risk):
    """The gate on every sequence: its block risks against its oracle's, the GPU's repairs equal
    to its oracle gate's on the GPU's risks and, outside the tie zone, on the oracle's own."""
    risk = rg.gpu.export(layer, _lib.X_BLOCK_RISK).cpu().numpy()
    before = [ref.repaired[layer][0].copy() for ref in rg.refs]
    rg.gpu.witcert_gate(layer, tau)
    slots = rg.gpu.export(layer, _lib.X_SLOTS).cpu().numpy()
    for i, ref in enumerate(rg.refs):
        nblk = (lens[i] + 15) // 16
        assert not np.any(risk[i, :, nblk:])
        check_risk(risk[i, :, :nblk], oracle_risk[i], what=f"block risk seq {i}")
        ref.gate(layer, tau, risk[i:i + 1, :, :nblk])
        np.testing.assert_array_equal(slots[i, :, :nblk] >= 0, ref.repaired[layer][0])
        assert check_gate_end_to_end(oracle_risk[i][None], before[i][None], tau, slots[i:i + 1, :, :nblk] >= 0,
                                     rg.w.group) == 0


WIDE_CASES = [
    ("int8_dither", 20, False, 4.0),   # CTAs of 16 sequences: a full one and one of 4; gated
    ("fp8_e4m3", 16, True, 0.5),       # one group, paged, gated
    ("kivi2", 9, False, None),         # CTAs of 8 sequences: a full one and one of a single sequence
    ("int8_rtn", 12, True, None),
    ("blackbox", 8, False, None),
]


@pytest.mark.parametrize("scheme,B,paged,tau", WIDE_CASES)
def test_wide_ragged_batches_match_each_sequence(scheme, B, paged, tau):
    """Ragged bf16 batches of 8 to 20 sequences: split CTAs of 8 and 16 warps, a full group of
    sequences and a partial one.  Lengths from 0 to 1500 (an empty sequence, a single token,
    equal lengths, ragged tails); every sequence against its own oracle, then one-token appends
    to every other sequence (some crossing a block boundary), a reset of the longest, and decodes
    again."""
    w = WORKLOADS["qwen_1l"].with_(batch=B, context=1500, steps=4, scheme=scheme)
    rng = np.random.default_rng(B)
    lens = [int(n) for n in rng.integers(2, 1501, B)]
    lens[0], lens[1], lens[2] = 0, 1, 1500
    lens[3] = lens[4] = lens[5] = lens[6] = lens[7] = 640      # ties across the first group's end
    lens[B - 1] = 32
    pages = sum((n + 16) // 16 + 1 for n in lens) + 8 if paged else 0
    gate = tau is not None
    rg = Ragged(w, scheme, cap=1536, v_witness=not gate, gate_blocks=B * 4 * 96 if gate else 0, max_pages=pages)
    K, V = gen_kv(w, 0)
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    rg.check_store(0)
    _, _, oracle_risk = rg.check_decode(0, gen_q(w, 0, 0), w.delta_req)
    if gate:
        _gate_check(rg, 0, tau, lens, oracle_risk)
    K2, V2 = gen_kv(w.with_(context=16), 3)
    app = [1 if i % 2 == 0 else 0 for i in range(B)]
    rg.write(0, list(zip(_split(K2, app), _split(V2, app))))
    lens = [n + a for n, a in zip(lens, app)]
    _, _, oracle_risk = rg.check_decode(0, gen_q(w, 0, 1), w.delta_req)
    if gate:
        _gate_check(rg, 0, tau, lens, oracle_risk)
    rg.gpu.witcert_reset_sequence(2)
    rg.refs[2] = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, 1, scheme, w.seed, w.steps, v_witness=not gate)
    rg.check_decode(0, gen_q(w, 0, 2), w.delta_req)
    assert rg.gpu.witcert_stats()["device_errors"] == 0


def test_ragged_rejects_overflow_and_partial_decode():
    w = WORKLOADS["tiny"].with_(batch=2)
    rg = Ragged(w, "int8_dither", cap=40)
    K, V = gen_kv(w, 0)
    with pytest.raises(wc.WitcertError) as e:
        rg.gpu.witcert_write_ragged(0, rg.dev(K[0, :41]), rg.dev(V[0, :41]), [41, 0])
    assert e.value.status == _lib.EINVAL
    assert rg.gpu.witcert_seq_length(0, 0) == 0
    rg.write(0, [(K[0, :10], V[0, :10]), (K[1, :3], V[1, :3])])
    with pytest.raises(wc.WitcertError) as e:
        rg.gpu.decode_partial(0, rg.dev(gen_q(w, 0, 0)), w.delta_req, 10)
    assert e.value.status == _lib.ESTATE


@pytest.mark.parametrize("scheme", ["int8_dither", "kivi2"])
def test_paged_uniform_writes_and_pool_exhaustion(scheme):
    """Equal appends to a paged cache take the batched writers through the page table; a write
    the pool cannot hold fails with ENOMEM and changes nothing; after a reset frees pages the
    same write succeeds.  Every result matches the oracle."""
    w = WORKLOADS["qwen_1l"].with_(batch=3, context=200, steps=2, scheme=scheme)
    rg = Ragged(w, scheme, cap=400, max_pages=3 * 13 + 5)
    K, V = gen_kv(w, 0)
    lens = [200, 200, 200]                      # 13 blocks each
    rg.write(0, list(zip(_split(K, lens), _split(V, lens))))
    assert rg.gpu.witcert_stats()["pages_used"] == 39
    rg.check_store(0)
    rg.check_decode(0, gen_q(w, 0, 0), w.delta_req)
    K2, V2 = gen_kv(w.with_(context=120), 4)
    big = [0, 120, 0]                           # blocks 13..19: 7 new pages > 5 free
    with pytest.raises(wc.WitcertError) as e:
        rg.gpu.witcert_write_ragged(0, rg.dev(K2[1, :120]), rg.dev(V2[1, :120]), big)
    assert e.value.status == _lib.ENOMEM
    assert rg.gpu.witcert_seq_length(0, 1) == 200 and rg.gpu.witcert_stats()["pages_used"] == 39
    rg.check_decode(0, gen_q(w, 0, 1), w.delta_req)
    rg.gpu.witcert_reset_sequence(0)
    rg.refs[0] = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, 1, scheme, w.seed, w.steps, v_witness=True)
    rg.write(0, list(zip(_split(K2, big), _split(V2, big))))
    assert rg.gpu.witcert_stats()["pages_used"] == 26 + 7
    rg.check_store(0)
    rg.check_decode(0, gen_q(w, 0, 1), w.delta_req)


def test_reset_clears_value_witnesses_of_the_last_block():
    """Black-box scheme: a sequence whose value witnesses overflowed to +inf (the caller's f(V)
    is 1e5 off in channel 0) is reset and refilled with 10 tokens.  Rows 10..15 of its last block
    are read with weight 0, so they must hold zero, not the stale +inf (0 x inf would make the
    value meter NaN)."""
    w = WORKLOADS["qwen_1l"].with_(batch=2, context=40, steps=2, scheme="blackbox")
    rg = Ragged(w, "blackbox", cap=64)
    K, V = gen_kv(w, 0)
    Kd, Vd = rg.dev(K[1, :40]), rg.dev(V[1, :40])
    Vh = V[1, :40].copy()
    Vh[..., 0] += 1e5
    rg.gpu.witcert_write_ragged(0, Kd, Vd, [0, 40], rg.dev(tensor_function(K[1, :40], 3)), rg.dev(Vh))
    wv = rg.gpu.export(0, _lib.X_V_WITNESS).cpu().numpy()
    assert np.all(np.isposinf(wv[1, :40]))
    rg.gpu.witcert_reset_sequence(1)
    rg.refs[1] = OracleCache(w.n_layers, w.n_q_heads, w.n_kv_heads, 1, "blackbox", w.seed, w.steps, v_witness=True)
    K2, V2 = gen_kv(w.with_(context=20), 4)
    rg.write(0, list(zip(_split(K2, [20, 10]), _split(V2, [20, 10]))))
    rg.check_store(0)
    wv = rg.gpu.export(0, _lib.X_V_WITNESS).cpu().numpy()
    assert not np.any(wv[1, 10:16])
    _, mm, _ = rg.check_decode(0, gen_q(w, 0, 0), w.delta_req)
    assert np.all(np.isfinite(mm["meter_v"]))
