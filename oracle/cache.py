"""Whole-path oracle: a cache that is written, decoded and gated like the library's.

Slow and plain: it keeps every layer's exact keys and values, quantizes each
appended token with the scheme's writer, and decodes every (sequence, KV head)
group with decode_ref over the full context (no splits).

KIVI keys are quantized per channel over 16-token blocks, so a block is
quantized when its 16th token arrives; until then its tokens stay exact
(witness 0), the way KIVI keeps its most recent tokens in full precision.

The black-box scheme takes the caller's tensor-function outputs K_hat, V_hat
with every write and keeps them as bfloat16.  With v_witness on, every scheme
also keeps one value witness per token and head and the decode reports the
value meter E_V.
"""
from __future__ import annotations

import numpy as np

from .gate import gate_group
from .meter import decode_ref, delta_loc
from .philox import dither
from .quant import (BLOCK, D, value_witness, witness, witness_stored, write_blackbox, write_fp8,
                    write_int8_dither, write_kivi2_k, write_kivi2_v)

SCHEMES = ("int8_dither", "fp8_e4m3", "kivi2", "int8_rtn", "blackbox")


class OracleCache:
    def __init__(self, n_layers, n_q_heads, n_kv_heads, batch, scheme, seed=0, total_steps=1, v_witness=False):
        assert scheme in SCHEMES
        self.L, self.Hq, self.Hkv, self.B = n_layers, n_q_heads, n_kv_heads, batch
        self.g = n_q_heads // n_kv_heads
        self.scheme, self.seed, self.T = scheme, seed, total_steps
        self.v_witness = bool(v_witness)
        shape0 = (batch, 0, n_kv_heads, D)
        self.k = [np.zeros(shape0, np.float32) for _ in range(n_layers)]     # exact keys
        self.v = [np.zeros(shape0, np.float32) for _ in range(n_layers)]
        self.khat = [np.zeros(shape0) for _ in range(n_layers)]
        self.vhat = [np.zeros(shape0) for _ in range(n_layers)]
        self.w64 = [np.zeros((batch, 0, n_kv_heads, 16)) for _ in range(n_layers)]
        self.w16 = [np.zeros((batch, 0, n_kv_heads, 16), np.float16) for _ in range(n_layers)]
        self.wv64 = [np.zeros((batch, 0, n_kv_heads)) for _ in range(n_layers)]
        self.wv16 = [np.zeros((batch, 0, n_kv_heads), np.float16) for _ in range(n_layers)]
        self.kcode = [np.zeros((batch, 0, n_kv_heads, D), np.int16) for _ in range(n_layers)]
        self.vcode = [np.zeros((batch, 0, n_kv_heads, D), np.int16) for _ in range(n_layers)]
        self.kscale = [np.zeros((batch, 0, n_kv_heads, 4), np.float16) for _ in range(n_layers)]
        self.vscale = [np.zeros((batch, 0, n_kv_heads, 4), np.float16) for _ in range(n_layers)]
        self.vzero = [np.zeros((batch, 0, n_kv_heads, 4), np.float16) for _ in range(n_layers)]
        self.kivi_kp = [dict() for _ in range(n_layers)]   # (seq, h, blk) -> (scale[128], zero[128])
        self.repaired = [np.zeros((batch, n_kv_heads, 0), bool) for _ in range(n_layers)]
        self.clamps = 0

    def length(self, layer):
        return self.k[layer].shape[1]

    # ------------------------------------------------------------------ write

    def write(self, layer, K, V, K_hat=None, V_hat=None):
        """Append K, V [B, n, Hkv, d] (float32 values exact in the input dtype); the black-box
        scheme also takes its tensor function's outputs K_hat, V_hat of the same shape."""
        K = np.asarray(K, np.float32)
        V = np.asarray(V, np.float32)
        assert (K_hat is not None) == (self.scheme == "blackbox")
        B, n, H, _ = K.shape
        t0 = self.length(layer)
        pos = np.arange(t0, t0 + n)
        kh = np.zeros((B, n, H, D))
        vh = np.zeros((B, n, H, D))
        kc = np.zeros((B, n, H, D), np.int16)
        vc = np.zeros((B, n, H, D), np.int16)
        ks = np.zeros((B, n, H, 4), np.float16)
        vs = np.zeros((B, n, H, 4), np.float16)
        vz = np.zeros((B, n, H, 4), np.float16)
        for h in range(H):
            if self.scheme in ("int8_dither", "int8_rtn"):
                # round to nearest is the dithered quantizer with xi = 0
                if self.scheme == "int8_dither":
                    xik = dither(self.seed, layer, h, pos, 0)
                    xiv = dither(self.seed, layer, h, pos, 1)
                else:
                    xik = xiv = np.zeros((n, D), np.float32)
                for i in range(B):
                    c, s, xh, cl = write_int8_dither(K[i, :, h], xik)
                    kc[i, :, h], ks[i, :, h], kh[i, :, h] = c, s, xh
                    self.clamps += cl
                    c, s, xh, cl = write_int8_dither(V[i, :, h], xiv)
                    vc[i, :, h], vs[i, :, h], vh[i, :, h] = c, s, xh
                    self.clamps += cl
            elif self.scheme == "blackbox":
                kh[:, :, h] = write_blackbox(np.asarray(K_hat, np.float32)[:, :, h].reshape(-1, D)).reshape(B, n, D)
                vh[:, :, h] = write_blackbox(np.asarray(V_hat, np.float32)[:, :, h].reshape(-1, D)).reshape(B, n, D)
            elif self.scheme == "fp8_e4m3":
                c, xh = write_fp8(K[:, :, h])
                kc[:, :, h], kh[:, :, h] = c, xh
                c, xh = write_fp8(V[:, :, h])
                vc[:, :, h], vh[:, :, h] = c, xh
            else:
                kh[:, :, h] = K[:, :, h]          # exact until the block completes
                for i in range(B):
                    c, s, z, xh = write_kivi2_v(V[i, :, h])
                    vc[i, :, h], vs[i, :, h], vz[i, :, h], vh[i, :, h] = c, s, z, xh
        self.k[layer] = np.concatenate([self.k[layer], K], 1)
        self.v[layer] = np.concatenate([self.v[layer], V], 1)
        self.khat[layer] = np.concatenate([self.khat[layer], kh], 1)
        self.vhat[layer] = np.concatenate([self.vhat[layer], vh], 1)
        self.kcode[layer] = np.concatenate([self.kcode[layer], kc], 1)
        self.vcode[layer] = np.concatenate([self.vcode[layer], vc], 1)
        self.kscale[layer] = np.concatenate([self.kscale[layer], ks], 1)
        self.vscale[layer] = np.concatenate([self.vscale[layer], vs], 1)
        self.vzero[layer] = np.concatenate([self.vzero[layer], vz], 1)
        wv = value_witness(V - vh)
        self.wv64[layer] = np.concatenate([self.wv64[layer], wv], 1)
        self.wv16[layer] = np.concatenate([self.wv16[layer], witness_stored(wv)], 1)
        w = witness(self.k[layer][:, t0:] - self.khat[layer][:, t0:])
        self.w64[layer] = np.concatenate([self.w64[layer], w], 1)
        self.w16[layer] = np.concatenate([self.w16[layer], witness_stored(w)], 1)
        if self.scheme == "kivi2":
            self._kivi_close_blocks(layer, t0, t0 + n)
        nblk = (self.length(layer) + BLOCK - 1) // BLOCK
        grow = nblk - self.repaired[layer].shape[2]
        if grow > 0:
            self.repaired[layer] = np.concatenate(
                [self.repaired[layer], np.zeros((B, H, grow), bool)], 2)

    def _kivi_close_blocks(self, layer, t0, t1):
        for blk in range(t0 // BLOCK, t1 // BLOCK):
            lo, hi = blk * BLOCK, (blk + 1) * BLOCK
            for i in range(self.B):
                for h in range(self.Hkv):
                    c, s, z, xh = write_kivi2_k(self.k[layer][i, lo:hi, h])
                    self.kcode[layer][i, lo:hi, h] = c
                    self.khat[layer][i, lo:hi, h] = xh
                    self.kivi_kp[layer][(i, h, blk)] = (s, z)
                    w = witness(self.k[layer][i, lo:hi, h] - xh)
                    self.w64[layer][i, lo:hi, h] = w
                    self.w16[layer][i, lo:hi, h] = witness_stored(w)

    # ------------------------------------------------------------------ decode

    def group_view(self, layer, i, h):
        """khat, vhat, stored witness, K scales, repaired mask of one (seq, KV head), repairs applied."""
        S = self.length(layer)
        rep_blk = self.repaired[layer][i, h]
        rep = np.repeat(rep_blk, BLOCK)[:S] if S else np.zeros(0, bool)
        kh = self.khat[layer][i, :, h].copy()
        kh[rep] = self.k[layer][i, rep, h]
        w = self.w16[layer][i, :, h].astype(np.float64)
        w[rep] = 0.0
        ks = self.kscale[layer][i, :, h].astype(np.float64) if self.scheme == "int8_dither" else None
        return kh, self.vhat[layer][i, :, h], w, ks, rep

    def value_witness_view(self, layer, i, h):
        """Stored value witnesses [S] of one (sequence, KV head) as float64."""
        return self.wv16[layer][i, :, h].astype(np.float64)

    def decode(self, layer, q, delta_req):
        """q: [B, Hq, d].  Returns per-(seq, q-head) outputs, meters and block risks."""
        q = np.asarray(q, np.float64)
        S = self.length(layer)
        dl = delta_loc(delta_req, self.L, self.Hq, self.T)
        nblk = (S + BLOCK - 1) // BLOCK
        out = np.zeros((self.B, self.Hq, D))
        ma, mb = np.zeros((self.B, self.Hq)), np.full((self.B, self.Hq), np.nan)
        ra, rb = np.zeros((self.B, self.Hq)), np.full((self.B, self.Hq), np.nan)
        risk = np.zeros((self.B, self.Hq, nblk))
        mv = np.zeros((self.B, self.Hq)) if self.v_witness else None
        for i in range(self.B):
            for h in range(self.Hkv):
                js = slice(h * self.g, (h + 1) * self.g)
                kh, vh, w, ks, rep = self.group_view(layer, i, h)
                wv = self.value_witness_view(layer, i, h) if self.v_witness else None
                r = decode_ref(q[i, js], kh, vh, w, ks, rep, dl, wv)
                out[i, js] = r["out"]
                if mv is not None:
                    mv[i, js] = r["meter_v"]
                ma[i, js], ra[i, js] = r["meter_a"], r["raw_a"]
                if r["meter_b"] is not None:
                    mb[i, js], rb[i, js] = r["meter_b"], r["raw_b"]
                risk[i, js] = r["risk"]
        return dict(out=out, meter_a=ma, meter_b=mb, raw_a=ra, raw_b=rb, risk=risk, meter_v=mv)

    # ------------------------------------------------------------------ gate

    def gate(self, layer, tau, risk):
        """Repair what the gate selects from the given block risks [B, Hq, nblk]."""
        risk = np.asarray(risk, np.float32)
        picked = []
        for i in range(self.B):
            for h in range(self.Hkv):
                js = slice(h * self.g, (h + 1) * self.g)
                sel = gate_group(risk[i, js], self.repaired[layer][i, h], tau)
                for b in sel:
                    self.repaired[layer][i, h, b] = True
                    picked.append((i, h, b))
        return picked
