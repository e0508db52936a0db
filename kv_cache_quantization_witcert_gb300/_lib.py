"""ctypes declarations of the C ABI in include/witcert.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwitcert.so")

OK, EINVAL, ENOMEM, ECUDA, ETIMEDOUT, EPAGEIN, ESTATE = 0, -1, -2, -3, -4, -5, -6
INT8_DITHER, FP8_E4M3, KIVI2, INT8_RTN, BLACKBOX = 0, 1, 2, 3, 4
F32, BF16 = 0, 1
(X_K_CODES, X_V_CODES, X_K_SCALES, X_V_SCALES, X_V_ZEROS, X_KIVI_K_SCALE, X_KIVI_K_ZERO, X_WITNESS,
 X_SLOTS, X_BLOCK_RISK, X_V_WITNESS) = range(11)

FAULT_BACKING_LOST = 1

SCHEMES = {"int8_dither": INT8_DITHER, "fp8_e4m3": FP8_E4M3, "kivi2": KIVI2, "int8_rtn": INT8_RTN,
           "blackbox": BLACKBOX}
STATUS_NAMES = {OK: "OK", EINVAL: "EINVAL", ENOMEM: "ENOMEM", ECUDA: "ECUDA", ETIMEDOUT: "ETIMEDOUT",
                EPAGEIN: "EPAGEIN", ESTATE: "ESTATE"}


class witcert_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("batch", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("scheme", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("total_steps", ctypes.c_int), ("n_splits", ctypes.c_int), ("max_repair_blocks", ctypes.c_int),
                ("pos_offset", ctypes.c_int), ("v_witness", ctypes.c_int), ("max_pages", ctypes.c_int)]


class witcert_gate_counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("cells_triggered", "blocks_selected", "blocks_paged_in",
                                                "bytes_paged_in", "blocks_dropped", "gate_calls")]


class witcert_stats_t(ctypes.Structure):
    _fields_ = [("tokens_written", ctypes.c_uint64), ("decode_calls", ctypes.c_uint64),
                ("int8_clamps", ctypes.c_uint64), ("device_errors", ctypes.c_uint64),
                ("decode_kernel_ms", ctypes.c_double), ("decode_kernel_launches", ctypes.c_uint64),
                ("last_n_splits", ctypes.c_int), ("pages_used", ctypes.c_uint64)]


_vp, _int, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_fp = ctypes.POINTER(ctypes.c_float)

SIGNATURES = {
    "witcert_create": [ctypes.POINTER(witcert_config), ctypes.POINTER(_vp)],
    "witcert_destroy": [_vp],
    "witcert_write": [_vp, _int, _vp, _vp, _int, _vp],
    "witcert_write_hat": [_vp, _int, _vp, _vp, _vp, _vp, _int, _vp],
    "witcert_write_ragged": [_vp, _int, _vp, _vp, _vp, _vp, ctypes.POINTER(ctypes.c_int32), _vp],
    "witcert_reset_sequence": [_vp, _int, _vp],
    "witcert_seq_length": [_vp, _int, _int, ctypes.POINTER(_int)],
    "witcert_decode": [_vp, _int, _vp, ctypes.c_double, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "witcert_decode_noalloc": [_vp, _int, _vp, ctypes.c_double, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "witcert_decode_partial": [_vp, _int, _vp, ctypes.c_double, ctypes.c_longlong, _vp, _vp],
    "witcert_merge_partials": [_vp, _int, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "witcert_gate": [_vp, _int, ctypes.c_float, _vp],
    "witcert_gate_stats": [_vp, ctypes.POINTER(witcert_gate_counters), _int],
    "witcert_stats": [_vp, ctypes.POINTER(witcert_stats_t)],
    "witcert_set_profiling": [_vp, _int],
    "witcert_set_launch_overlap": [_vp, _int],
    "witcert_length": [_vp, _int, ctypes.POINTER(_int)],
    "witcert_export": [_vp, _int, _int, _vp, _sz, _vp],
    "witcert_dither": [ctypes.c_uint64, _int, _int, _int, _int, _int, _vp, _vp],
    "witcert_wait_selftest": [ctypes.c_int64, _vp],
    "witcert_gate_select": [_vp, _vp, _int, _int, _int, _int, ctypes.c_float, _vp, _vp],
    "witcert_inject_fault": [_vp, _int, _int],
    "witcert_quotient_selftest": [_int, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64), _vp],
    "witcert_last_error": [],
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libwitcert.so; raise if it has not been built (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m kv_cache_quantization_witcert_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name == "witcert_last_error" else ctypes.c_int
        _lib = lib
    return _lib


class WitcertError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().witcert_last_error().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise WitcertError(status, where)
