"""Python binding of libwitcert (GB300 metered KV-cache decode).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  Function names follow
the C ABI (include/witcert.h): witcert_create / write / decode / gate / ...
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (BF16, BLACKBOX, EINVAL, ENOMEM, EPAGEIN, ESTATE, ETIMEDOUT, F32, FP8_E4M3, INT8_DITHER,  # noqa: F401
                   INT8_RTN, KIVI2, SCHEMES, WitcertError, check, load)

__all__ = ["Cache", "witcert_dither", "witcert_merge_partials", "witcert_gate_select", "WitcertError", "load", "SCHEMES", "PART_STRIDE"]

_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _extent(t, i):
    """Extent i of a tensor argument, or None when it has none (_need then rejects it)."""
    return t.shape[i] if isinstance(t, torch.Tensor) and t.dim() > i else None


def _need(*specs):
    """Check the tensors a call hands the library, each spec (name, tensor, dtype, shape[,
    optional]) with None in shape for any extent: contiguous tensors of that dtype and shape,
    then all on a CUDA device.  The C ABI takes bare pointers, so a host tensor or a short
    buffer would reach a kernel; the binding raises ValueError instead."""
    given = []
    for name, t, dtype, shape, *opt in specs:
        if t is None:
            if opt and opt[0]:
                continue
            raise ValueError(f"{name} must not be None")
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if t.dim() != len(shape) or any(e is not None and e != x for e, x in zip(shape, t.shape)):
            want = tuple("*" if e is None else e for e in shape)
            raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")
        given.append((name, t))
    for name, t in given:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


class Cache:
    """One WitCert cache: compressed K/V store, witnesses, optional gate state."""

    def __init__(self, n_layers, n_q_heads, n_kv_heads, batch, max_tokens, scheme="int8_dither",
                 dtype=torch.bfloat16, seed=0, total_steps=1, n_splits=0, max_repair_blocks=0, pos_offset=0,
                 v_witness=False, max_pages=0):
        lib = load()
        self.dtype = dtype
        self.cfg = _lib.witcert_config(n_layers, n_q_heads, n_kv_heads, 128, batch, max_tokens,
                                       SCHEMES[scheme] if isinstance(scheme, str) else scheme,
                                       BF16 if dtype == torch.bfloat16 else F32, seed, total_steps, n_splits,
                                       max_repair_blocks, pos_offset, int(bool(v_witness)), max_pages)
        self.scheme = scheme
        self.v_witness = bool(v_witness)
        h = ctypes.c_void_p()
        check(lib.witcert_create(ctypes.byref(self.cfg), ctypes.byref(h)), "witcert_create")
        self._h = h

    # ------------------------------------------------------------------ ABI calls
    def _kv_shape(self, n_tok=None):
        return (self.cfg.batch, n_tok, self.cfg.n_kv_heads, 128)

    def _q_shape(self, last=128):
        return (self.cfg.batch, self.cfg.n_q_heads, last)

    def _decode_args(self, q, out, meters):
        names = ("meter_a", "meter_b", "raw_a", "raw_b", "meter_v")
        _need(("q", q, self.dtype, self._q_shape()), ("out", out, torch.float32, self._q_shape()),
              *((n, m, torch.float32, self._q_shape()[:2], True) for n, m in zip(names, meters)))

    def witcert_write(self, layer, K, V, stream=None):
        """Append K, V [batch, n_tok, n_kv_heads, 128] to every sequence of `layer`."""
        n_tok = _extent(K, 1)
        _need(("K", K, self.dtype, self._kv_shape(n_tok)), ("V", V, self.dtype, self._kv_shape(n_tok)))
        check(load().witcert_write(self._h, layer, _ptr(K), _ptr(V), n_tok, _stream_ptr(stream)), "witcert_write")

    def witcert_write_hat(self, layer, K, V, K_hat, V_hat, stream=None):
        """Black-box scheme: K_hat, V_hat are the tensor function's outputs f(K), f(V)."""
        n_tok = _extent(K, 1)
        _need(*((name, t, self.dtype, self._kv_shape(n_tok)) for name, t in
                (("K", K), ("V", V), ("K_hat", K_hat), ("V_hat", V_hat))))
        check(load().witcert_write_hat(self._h, layer, _ptr(K), _ptr(V), _ptr(K_hat), _ptr(V_hat), n_tok,
                                       _stream_ptr(stream)), "witcert_write_hat")

    def witcert_write_ragged(self, layer, K, V, n_tok, K_hat=None, V_hat=None, stream=None):
        """Ragged append: n_tok[i] tokens to sequence i; K, V (and K_hat, V_hat for black-box
        caches) packed sequence by sequence, [sum(n_tok), Hkv, 128]."""
        counts = [int(x) for x in n_tok]
        if len(counts) != self.cfg.batch:
            raise ValueError(f"n_tok needs one count per sequence ({self.cfg.batch}), got {len(counts)}")
        shape = (sum(counts), self.cfg.n_kv_heads, 128)
        _need(("K", K, self.dtype, shape), ("V", V, self.dtype, shape), ("K_hat", K_hat, self.dtype, shape, True),
              ("V_hat", V_hat, self.dtype, shape, True))
        arr = (ctypes.c_int32 * len(counts))(*counts)
        check(load().witcert_write_ragged(self._h, layer, _ptr(K), _ptr(V), _ptr(K_hat), _ptr(V_hat), arr,
                                          _stream_ptr(stream)), "witcert_write_ragged")

    def witcert_reset_sequence(self, seq, stream=None):
        check(load().witcert_reset_sequence(self._h, int(seq), _stream_ptr(stream)), "witcert_reset_sequence")

    def witcert_seq_length(self, layer, seq):
        n = ctypes.c_int()
        check(load().witcert_seq_length(self._h, layer, int(seq), ctypes.byref(n)), "witcert_seq_length")
        return n.value

    def witcert_decode(self, layer, q, delta_req, out, meter_a=None, meter_b=None, raw_a=None, raw_b=None,
                       meter_v=None, stream=None):
        self._decode_args(q, out, (meter_a, meter_b, raw_a, raw_b, meter_v))
        check(load().witcert_decode(self._h, layer, _ptr(q), float(delta_req), _ptr(out), _ptr(meter_a),
                                    _ptr(meter_b), _ptr(raw_a), _ptr(raw_b), _ptr(meter_v), _stream_ptr(stream)),
              "witcert_decode")

    def witcert_decode_noalloc(self, layer, q, delta_req, out, meter_a=None, meter_b=None, raw_a=None, raw_b=None,
                               meter_v=None, stream=None):
        self._decode_args(q, out, (meter_a, meter_b, raw_a, raw_b, meter_v))
        check(load().witcert_decode_noalloc(self._h, layer, _ptr(q), float(delta_req), _ptr(out), _ptr(meter_a),
                                            _ptr(meter_b), _ptr(raw_a), _ptr(raw_b), _ptr(meter_v),
                                            _stream_ptr(stream)), "witcert_decode_noalloc")

    def witcert_decode_partial(self, layer, q, delta_req, s_total, part, stream=None):
        _need(("q", q, self.dtype, self._q_shape()), ("part", part, torch.float32, self._q_shape(PART_STRIDE)))
        check(load().witcert_decode_partial(self._h, layer, _ptr(q), float(delta_req), int(s_total), _ptr(part),
                                            _stream_ptr(stream)), "witcert_decode_partial")

    def decode_partial(self, layer, q, delta_req, s_total, stream=None):
        """This shard's per-cell records [B, Hq, 136] (see witcert_decode_partial)."""
        part = torch.empty((q.shape[0], q.shape[1], PART_STRIDE), dtype=torch.float32, device=q.device)
        self.witcert_decode_partial(layer, q, delta_req, s_total, part, stream=stream)
        return part

    def witcert_gate(self, layer, tau, stream=None):
        check(load().witcert_gate(self._h, layer, float(tau), _stream_ptr(stream)), "witcert_gate")

    def witcert_inject_fault(self, fault, layer):
        """Host-side fault injection (see witcert_inject_fault in include/witcert.h)."""
        check(load().witcert_inject_fault(self._h, int(fault), int(layer)), "witcert_inject_fault")

    def witcert_gate_stats(self, timeout_ms=10000):
        s = _lib.witcert_gate_counters()
        check(load().witcert_gate_stats(self._h, ctypes.byref(s), timeout_ms), "witcert_gate_stats")
        return {f: getattr(s, f) for f, _ in s._fields_}

    def witcert_stats(self):
        s = _lib.witcert_stats_t()
        check(load().witcert_stats(self._h, ctypes.byref(s)), "witcert_stats")
        return {f: getattr(s, f) for f, _ in s._fields_}

    def witcert_set_profiling(self, on):
        check(load().witcert_set_profiling(self._h, int(bool(on))), "witcert_set_profiling")

    def witcert_set_launch_overlap(self, on):
        check(load().witcert_set_launch_overlap(self._h, int(bool(on))), "witcert_set_launch_overlap")

    def witcert_length(self, layer):
        n = ctypes.c_int()
        check(load().witcert_length(self._h, layer, ctypes.byref(n)), "witcert_length")
        return n.value

    def witcert_export(self, layer, what, dst, stream=None):
        _need(("dst", dst, getattr(dst, "dtype", None), tuple(getattr(dst, "shape", ()))))   # the library checks the size
        check(load().witcert_export(self._h, layer, what, _ptr(dst), dst.numel() * dst.element_size(),
                                    _stream_ptr(stream)), "witcert_export")

    def close(self):
        if getattr(self, "_h", None):
            check(load().witcert_destroy(self._h), "witcert_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ conveniences (allocation + the calls above)
    def decode(self, layer, q, delta_req, meters=True, stream=None):
        B, Hq = q.shape[0], q.shape[1]
        out = torch.empty((B, Hq, 128), dtype=torch.float32, device=q.device)
        if not meters:
            self.witcert_decode(layer, q, delta_req, out, stream=stream)
            return out, None
        m = torch.empty((5, B, Hq), dtype=torch.float32, device=q.device)
        self.witcert_decode(layer, q, delta_req, out, m[0], m[1], m[2], m[3], m[4] if self.v_witness else None,
                            stream=stream)
        meters = {"meter_a": m[0], "meter_b": m[1], "raw_a": m[2], "raw_b": m[3]}
        if self.v_witness:
            meters["meter_v"] = m[4]
        return out, meters

    def export(self, layer, what, stream=None):
        B, Hkv, Hq = self.cfg.batch, self.cfg.n_kv_heads, self.cfg.n_q_heads
        S = self.witcert_length(layer)
        nblk = (S + 15) // 16
        dev = torch.device("cuda", torch.cuda.current_device())
        code_dt = torch.bfloat16 if self.cfg.scheme == BLACKBOX else torch.uint8
        shapes = {
            _lib.X_K_CODES: ((B, S, Hkv, 128), code_dt), _lib.X_V_CODES: ((B, S, Hkv, 128), code_dt),
            _lib.X_K_SCALES: ((B, S, Hkv, 4), torch.float16), _lib.X_V_SCALES: ((B, S, Hkv, 4), torch.float16),
            _lib.X_V_ZEROS: ((B, S, Hkv, 4), torch.float16),
            _lib.X_KIVI_K_SCALE: ((B, nblk, Hkv, 128), torch.float16),
            _lib.X_KIVI_K_ZERO: ((B, nblk, Hkv, 128), torch.float16),
            _lib.X_WITNESS: ((B, S, Hkv, 16), torch.float16), _lib.X_SLOTS: ((B, Hkv, nblk), torch.int32),
            _lib.X_BLOCK_RISK: ((B, Hq, nblk), torch.float32), _lib.X_V_WITNESS: ((B, S, Hkv), torch.float16),
        }
        shape, dt = shapes[what]
        dst = torch.empty(shape, dtype=dt, device=dev)
        if dst.numel():
            self.witcert_export(layer, what, dst, stream=stream)
        return dst


PART_STRIDE = 136     # floats per (sequence, query head) record: m, Z, S_A, S_B, S_V, 3 unused, 128 value sums


def witcert_merge_partials(parts, scheme, out=None, meters=True, stream=None):
    """Merge shard records parts [B, Hq, n_parts, 136] (device fp32) into the output [B, Hq, 128]
    and, with meters, {"meter_a", "meter_b", "raw_a", "raw_b", "meter_v"} (see witcert_merge_partials)."""
    _need(("parts", parts, torch.float32, (None, None, None, PART_STRIDE)))
    B, Hq, n = parts.shape[0], parts.shape[1], parts.shape[2]
    if out is None:
        out = torch.empty((B, Hq, 128), dtype=torch.float32, device=parts.device)
    _need(("out", out, torch.float32, (B, Hq, 128)))
    m = torch.empty((5, B, Hq), dtype=torch.float32, device=parts.device) if meters else None
    ptrs = tuple(_ptr(m[k]) for k in range(5)) if meters else (None,) * 5
    check(load().witcert_merge_partials(_ptr(parts), n, B, Hq, SCHEMES[scheme] if isinstance(scheme, str) else scheme,
                                        _ptr(out), *ptrs, _stream_ptr(stream)), "witcert_merge_partials")
    return out, ({"meter_a": m[0], "meter_b": m[1], "raw_a": m[2], "raw_b": m[3], "meter_v": m[4]}
                 if meters else None)


def witcert_gate_select(risk, n_kv_heads, tau, repaired=None, selected=None, stream=None):
    """The gate's block selection on caller arrays: risk [B, Hq, nblk] float32 (device), repaired
    [B, Hkv, nblk] uint8 or None; returns the selection bitmap [B, Hkv, nblk // 32 + 1] int32
    (see witcert_gate_select)."""
    _need(("risk", risk, torch.float32, (None, None, None)))
    B, Hq, nblk = risk.shape
    _need(("repaired", repaired, torch.uint8, (B, n_kv_heads, nblk), True))
    if selected is None:
        selected = torch.empty((B, n_kv_heads, nblk // 32 + 1), dtype=torch.int32, device=risk.device)
    _need(("selected", selected, torch.int32, (B, n_kv_heads, nblk // 32 + 1)))
    check(load().witcert_gate_select(_ptr(risk), _ptr(repaired), B, Hq, n_kv_heads, nblk, float(tau), _ptr(selected),
                                     _stream_ptr(stream)), "witcert_gate_select")
    return selected


def witcert_quotient_selftest(n_f32=4096, seed=0, stream=None):
    """Differing quotients between the writers' x / s and the IEEE quotient over every positive
    fp16 scale (see witcert_quotient_selftest); expected 0."""
    n = ctypes.c_uint64()
    check(load().witcert_quotient_selftest(int(n_f32), int(seed), ctypes.byref(n), _stream_ptr(stream)),
          "witcert_quotient_selftest")
    return n.value


def witcert_wait_selftest(limit_ns, stream=None):
    """Run the bounded device wait against a barrier nothing completes; returns the status code."""
    return load().witcert_wait_selftest(int(limit_ns), _stream_ptr(stream))


def witcert_dither(seed, layer, kv_head, t0, n, tensor, out=None, stream=None):
    """Device dither xi [n, 128] float32 (see witcert_dither in include/witcert.h)."""
    if out is None:
        out = torch.empty((n, 128), dtype=torch.float32, device="cuda")
    _need(("out", out, torch.float32, (n, 128)))
    check(load().witcert_dither(seed, layer, kv_head, t0, n, tensor, _ptr(out), _stream_ptr(stream)),
          "witcert_dither")
    return out
