"""Synthetic KV-cache workloads (numpy PCG64, seeded).

The pages measure on Qwen2.5-7B, Mistral-7B and Yi-1.5-6B activations and on
RULER/LongBench prompts; none of those are available here, so these draws stand
in for them with the same shapes and the same structure the pages point at:

* keys and values ~ N(0, 1) per channel;
* "massive activation" outlier key channels, scaled before RoPE, placed on
  whole RoPE rotation pairs (dims i and i+64 under the rotate-half layout);
* RoPE applied to keys with the model's base (1e4, 1e6 or 5e6), so the cache
  holds post-RoPE keys as a serving system does;
* one planted high-score key per sequence ("needle"): at a seeded position the
  post-RoPE key of every KV head is c*n (n a random unit vector), and every
  query of that head's group is a*n + N(0, I), with a*c/sqrt(d) = 8;
* values rounded to bf16 (or kept fp32 for the tiny case).

Nothing here quantizes, measures or gates anything.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

HEAD_DIM = 128
_PLANT_LOGIT = 8.0  # a*c/sqrt(d) for the planted key


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    batch: int
    context: int
    steps: int
    dtype: str                 # "f32" or "bf16": dtype of K, V and q
    rope_base: float
    outlier_dims: tuple        # pre-RoPE key dims that carry outliers
    outlier_scale: float
    planted: bool
    scheme: str                # "int8_dither", "fp8_e4m3" or "kivi2"
    delta_req: float = 1e-2
    n_splits: int = 0          # 0 = let the library choose
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 1 layer, GQA 2, 256 cached tokens, 4 decode steps, fp32 inputs.
    "tiny": Workload("tiny", 1, 4, 2, 1, 256, 4, "f32", 1e4, (10, 11, 74, 75), 20.0,
                     False, "int8_dither", 1e-2, 0, 0),
    # Qwen2.5-7B-shaped single layer: 28q/4kv, B=8 x 4096, 64 steps.
    "qwen_1l": Workload("qwen_1l", 1, 28, 4, 8, 4096, 64, "bf16", 1e6, (10, 74), 50.0,
                        True, "int8_dither", 1e-2, 0, 0),
    # Full 28-layer Qwen2.5-7B-shaped decode, B=16 x 4096, 8 KV splits.
    "qwen_28l": Workload("qwen_28l", 28, 28, 4, 16, 4096, 64, "bf16", 1e6, (10, 74), 50.0,
                         True, "int8_dither", 1e-2, 8, 0),
    # Gated repair: Qwen 28L, B=8 x 32768, raw-cast FP8, 256 steps.
    "gated": Workload("gated", 28, 28, 4, 8, 32768, 256, "bf16", 1e6, (10, 74), 50.0,
                      True, "fp8_e4m3", 1e-2, 0, 0),
}

_SWEEP_SHAPES = {
    "mistral": dict(n_q_heads=32, n_kv_heads=8, rope_base=1e4),
    "yi": dict(n_q_heads=32, n_kv_heads=4, rope_base=5e6),
}


def sweep_workload(model: str, batch: int, context: int, scheme: str = "int8_dither",
                   n_layers: int = 32) -> Workload:
    """Long-context bandwidth sweep point (Mistral-7B or Yi-1.5-6B shaped)."""
    shp = _SWEEP_SHAPES[model]
    return Workload(f"{model}_b{batch}_s{context}", n_layers, shp["n_q_heads"], shp["n_kv_heads"],
                    batch, context, 1, "bf16", shp["rope_base"], (10, 74), 50.0, True, scheme,
                    1e-2, 0, 0)


# --------------------------------------------------------------------------- dtype rounding

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # finite inputs stay below 2^32 after adding at most 0x8000
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 array holding the bf16-rounded values."""
    return bf16_from_bits(bf16_bits(x))


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return bf16_round(x) if dtype == "bf16" else x


# --------------------------------------------------------------------------- RNG streams

_TAG_KV, _TAG_Q, _TAG_PLANT, _TAG_APPEND = 1, 2, 3, 4


def _rng(w: Workload, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, *tags])))


def _rope_tables(positions: np.ndarray, base: float, d: int = HEAD_DIM):
    half = d // 2
    inv = base ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = positions.astype(np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _apply_rope(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE on the last axis; x is [B, S, H, d], positions is [S]."""
    cos, sin = _rope_tables(positions, base, x.shape[-1])
    cos = cos[None, :, None, :]
    sin = sin[None, :, None, :]
    half = x.shape[-1] // 2
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def _plant(w: Workload, layer: int):
    """Per (seq): planted position; per (seq, kv head): unit direction n."""
    rng = _rng(w, _TAG_PLANT, layer)
    pos = rng.integers(0, w.context, size=w.batch)
    n = rng.standard_normal((w.batch, w.n_kv_heads, HEAD_DIM))
    n /= np.linalg.norm(n, axis=-1, keepdims=True)
    amp = math.sqrt(_PLANT_LOGIT * math.sqrt(HEAD_DIM))   # a = c, a*c/sqrt(d) = 8
    return pos, n.astype(np.float32), amp


def planted_positions(w: Workload, layer: int) -> np.ndarray:
    return _plant(w, layer)[0] if w.planted else np.full(w.batch, -1)


def _draw_keys(w: Workload, rng: np.random.Generator, n_seq: int, positions: np.ndarray):
    k = rng.standard_normal((n_seq, len(positions), w.n_kv_heads, HEAD_DIM), dtype=np.float32)
    if w.outlier_dims:
        k[..., list(w.outlier_dims)] *= np.float32(w.outlier_scale)
    return _apply_rope(k, positions, w.rope_base)


def gen_kv(w: Workload, layer: int):
    """Prefill K, V of one layer: float32 arrays [B, context, Hkv, d], exact in w.dtype."""
    rng = _rng(w, _TAG_KV, layer)
    pos = np.arange(w.context)
    k = _draw_keys(w, rng, w.batch, pos)
    v = rng.standard_normal((w.batch, w.context, w.n_kv_heads, HEAD_DIM), dtype=np.float32)
    if w.planted:
        ppos, n, amp = _plant(w, layer)
        for i in range(w.batch):
            k[i, ppos[i]] = amp * n[i]
    return _to_dtype(k, w.dtype), _to_dtype(v, w.dtype)


def gen_append_kv(w: Workload, layer: int, step: int):
    """K, V of the token appended at decode step `step` (position context+step): [B, 1, Hkv, d]."""
    rng = _rng(w, _TAG_APPEND, layer, step)
    pos = np.array([w.context + step])
    k = _draw_keys(w, rng, w.batch, pos)
    v = rng.standard_normal((w.batch, 1, w.n_kv_heads, HEAD_DIM), dtype=np.float32)
    return _to_dtype(k, w.dtype), _to_dtype(v, w.dtype)


def gen_q(w: Workload, layer: int, step: int):
    """Post-RoPE queries of one decode step: float32 [B, Hq, d], exact in w.dtype.

    Queries are drawn independently of everything stored in the cache (the
    non-adaptive regime of the pages' probabilistic certificate).
    """
    rng = _rng(w, _TAG_Q, layer, step)
    q = rng.standard_normal((w.batch, w.n_q_heads, HEAD_DIM), dtype=np.float32)
    if w.planted:
        _, n, amp = _plant(w, layer)
        kv_of = np.arange(w.n_q_heads) // w.group
        q += amp * n[:, kv_of, :]
    return _to_dtype(q, w.dtype)
