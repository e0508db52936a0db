"""Decode side of the oracle: attention, the two meter tiers, TV aggregation,
split-KV partial states and their log-sum-exp merge.  Plain float64 numpy.

Notation (per sequence, layer, decode step and query head):
    l~_t  = q . k^_t / sqrt(d)               logits against the compressed keys
    p~    = softmax(l~)                      compressed attention
    eps_t <= (1/sqrt d) sum_b ||q_b|| w_t,b  Tier A [WitCert summary, Theorem 2]
    s2_t  = (1/d) sum_c q_c^2 s_{c,t}^2 / 12
    u_t   = sqrt(2 s2_t log(2S/delta_loc))   Tier B [WitCert summary, Tier B paragraph]
    delta_loc = delta_req / (L*H*T)          H = query heads, T = decode steps
    A     = sum_t p~_t exp(c_t),  meter = min(1, (A^2 - 1)/2)
                                             [WitCert summary, improvements list: TV bound]
with c_t = eps_t (Tier A) or u_t (Tier B).  The oracle evaluates A as 1 + D with
D = sum_t p~_t expm1(c_t), and (A^2 - 1)/2 as D + D^2/2: the same numbers,
without the cancellation of A^2 - 1 when every c_t is small.

Value side (a reading of this library; the pages define no value bound): with the
stored value witness wv_t >= ||v_t - v^_t||,
    E_V = sum_t p~_t wv_t >= || sum_t p~_t v_t - sum_t p~_t v^_t ||
by the triangle inequality: the output error the value compression adds at the
compressed attention weights.
"""
from __future__ import annotations

import math

import numpy as np

from .quant import BAND_DIMS, BLOCK, D, GROUP


def delta_loc(delta_req: float, n_layers: int, n_q_heads: int, total_steps: int) -> float:
    """Request budget split over layers, query heads and decode steps [WitCert summary, Tier B]."""
    return delta_req / (n_layers * n_q_heads * total_steps)


def band_norms(q) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    return np.sqrt(np.sum(q[..., BAND_DIMS] ** 2, axis=-1))


def tier_a(q, w) -> np.ndarray:
    """eps[j, t] = (1/sqrt d) sum_b ||q_jb|| w_tb.   q: [g, d]; w: [S, 16]."""
    return band_norms(q) @ np.asarray(w, dtype=np.float64).T / math.sqrt(D)


def tier_b(q, k_scales, S: int, dloc: float) -> np.ndarray:
    """u[j, t] = sqrt(2 s2 log(2S/delta_loc)), s2 = (1/d) sum_c q_c^2 s_{c,t}^2 / 12.

    q: [g, d]; k_scales: [S, d/32] (one scale per 32-channel group of token t).
    """
    q = np.asarray(q, dtype=np.float64)
    s = np.repeat(np.asarray(k_scales, dtype=np.float64), GROUP, axis=-1)   # s_{c,t}: [S, d]
    s2 = (q ** 2) @ (s ** 2).T / (12.0 * D)                                  # [g, S]
    return np.sqrt(2.0 * s2 * math.log(2.0 * S / dloc))


def softmax(x, axis=-1):
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention(q, k, v):
    """Plain softmax attention: logits q.k/sqrt(d), weights, output.  q [g,d], k/v [S,d]."""
    logits = np.asarray(q, np.float64) @ np.asarray(k, np.float64).T / math.sqrt(D)
    p = softmax(logits)
    return logits, p, p @ np.asarray(v, np.float64)


def tv_meter(p_tilde, c):
    """(meter, raw, D) with A = sum p~ e^c = 1 + D and raw = (A^2 - 1)/2 = D + D^2/2."""
    Dv = np.sum(np.asarray(p_tilde) * np.expm1(np.asarray(c, np.float64)), axis=-1)
    raw = Dv + 0.5 * Dv * Dv
    return np.minimum(1.0, raw), raw, Dv


def value_meter(p_tilde, wv) -> np.ndarray:
    """E_V = sum_t p~_t wv_t.   p_tilde: [g, S]; wv: [S] stored value witnesses."""
    return np.asarray(p_tilde, np.float64) @ np.asarray(wv, np.float64)


def tv_exact(p, p_tilde) -> np.ndarray:
    """Total variation between exact and compressed attention: (1/2) sum_t |p_t - p~_t|."""
    return 0.5 * np.sum(np.abs(np.asarray(p) - np.asarray(p_tilde)), axis=-1)


def block_risk(p_tilde, c, S: int) -> np.ndarray:
    """Per-block share of D: R_blk = sum_{t in blk} p~_t expm1(c_t), 16-token blocks."""
    terms = np.asarray(p_tilde) * np.expm1(np.asarray(c, np.float64))
    nblk = (S + BLOCK - 1) // BLOCK
    pad = nblk * BLOCK - S
    terms = np.concatenate([terms, np.zeros(terms.shape[:-1] + (pad,))], axis=-1)
    return terms.reshape(terms.shape[:-1] + (nblk, BLOCK)).sum(-1)


def decode_ref(q, khat, vhat, w, k_scales=None, repaired=None, dloc=None, wv=None):
    """Metered decode of one (sequence, KV head) group over its whole context.

    q: [g, d] query heads of the group; khat/vhat: [S, d] keys/values the decode
    attends to (dequantized, or exact for repaired tokens); w: [S, 16] witness
    (zero for repaired tokens); k_scales: [S, 4] INT8 key scales (dither scheme
    only, enables Tier B); repaired: [S] bool; wv: [S] value witnesses (enables
    the value meter E_V).
    """
    q = np.asarray(q, dtype=np.float64)
    S = khat.shape[0]
    g = q.shape[0]
    if S == 0:
        z = np.zeros(g)
        return dict(out=np.zeros((g, D)), p=np.zeros((g, 0)), eps=np.zeros((g, 0)), u=None,
                    meter_a=z, raw_a=z, D_a=z, meter_b=z if k_scales is not None else None,
                    raw_b=z if k_scales is not None else None, D_b=z if k_scales is not None else None,
                    meter_v=z if wv is not None else None, risk=np.zeros((g, 0)))
    rep = np.zeros(S, bool) if repaired is None else np.asarray(repaired, bool)
    _, p, out = attention(q, khat, vhat)
    eps = tier_a(q, w)
    eps[:, rep] = 0.0
    meter_a, raw_a, D_a = tv_meter(p, eps)
    res = dict(out=out, p=p, eps=eps, u=None, meter_a=meter_a, raw_a=raw_a, D_a=D_a,
               meter_b=None, raw_b=None, D_b=None,
               meter_v=value_meter(p, wv) if wv is not None else None)
    c_gate = eps
    if k_scales is not None:
        u = tier_b(q, k_scales, S, dloc)
        u[:, rep] = 0.0
        meter_b, raw_b, D_b = tv_meter(p, u)
        res.update(u=u, meter_b=meter_b, raw_b=raw_b, D_b=D_b)
        c_gate = u
    res["risk"] = block_risk(p, c_gate, S)
    return res


# --------------------------------------------------------------------------- split-KV states

def partial_state(q, khat, vhat, c_a, c_b, lo: int, hi: int, wv=None):
    """Unnormalized state of tokens [lo, hi): running max m, Z = sum e^(l-m),
    S_X = sum e^(l-m) expm1(c_X), S_V = sum e^(l-m) wv, acc = sum e^(l-m) v^
    [WitCert summary, implementation: LSE-merged certificate accumulation across
    KV splits]."""
    q = np.asarray(q, np.float64)
    g = q.shape[0]
    wv = np.zeros(khat.shape[0]) if wv is None else np.asarray(wv, np.float64)
    if hi <= lo:
        return dict(m=np.full(g, -np.inf), Z=np.zeros(g), SA=np.zeros(g), SB=np.zeros(g),
                    SV=np.zeros(g), acc=np.zeros((g, D)))
    logits = q @ np.asarray(khat[lo:hi], np.float64).T / math.sqrt(D)
    m = logits.max(-1)
    e = np.exp(logits - m[:, None])
    return dict(m=m, Z=e.sum(-1), SA=(e * np.expm1(c_a[:, lo:hi])).sum(-1),
                SB=(e * np.expm1(c_b[:, lo:hi])).sum(-1), SV=e @ wv[lo:hi],
                acc=e @ np.asarray(vhat[lo:hi], np.float64))


def merge_states(states):
    """Log-sum-exp merge of split states: rescale each by e^(m_s - M), sum, normalize."""
    M = np.max(np.stack([s["m"] for s in states]), axis=0)
    Z = np.zeros_like(M)
    SA = np.zeros_like(M)
    SB = np.zeros_like(M)
    SV = np.zeros_like(M)
    acc = np.zeros(M.shape + (D,))
    for s in states:
        f = np.where(np.isfinite(s["m"]), np.exp(s["m"] - np.where(np.isfinite(M), M, 0.0)), 0.0)
        Z += f * s["Z"]
        SA += f * s["SA"]
        SB += f * s["SB"]
        SV += f * s["SV"]
        acc += f[:, None] * s["acc"]
    DA = SA / Z
    DB = SB / Z
    return dict(out=acc / Z[:, None], D_a=DA, D_b=DB, meter_a=np.minimum(1.0, DA + 0.5 * DA * DA),
                meter_b=np.minimum(1.0, DB + 0.5 * DB * DB), meter_v=SV / Z)
