"""The C-ABI library builds, loads and exports every function include/witcert.h declares (no GPU needed)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "witcert.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(witcert_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from kv_cache_quantization_witcert_gb300 import build
    try:
        return build.build()
    except RuntimeError as e:  # no toolkit on this machine
        pytest.skip(str(e))


def test_every_declared_symbol_is_exported(lib_path):
    names = _declared()
    assert len(names) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (witcert_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_library_loads_and_binding_matches_header(lib_path):
    import kv_cache_quantization_witcert_gb300 as w
    from kv_cache_quantization_witcert_gb300 import _lib
    lib = w.load()
    for n in _declared():
        assert hasattr(lib, n)
        assert n in _lib.SIGNATURES, f"binding lacks {n}"
    assert lib.witcert_last_error() == b""


def test_invalid_config_is_rejected_without_touching_the_gpu(lib_path):
    import ctypes

    import kv_cache_quantization_witcert_gb300 as w
    from kv_cache_quantization_witcert_gb300 import _lib
    lib = w.load()
    h = ctypes.c_void_p()
    bad = _lib.witcert_config(1, 4, 2, 64, 1, 16, 0, 0, 0, 1, 0, 0)          # head_dim 64
    assert lib.witcert_create(ctypes.byref(bad), ctypes.byref(h)) == _lib.EINVAL
    assert b"head_dim" in lib.witcert_last_error()
    bad = _lib.witcert_config(1, 36, 2, 128, 1, 16, 0, 0, 0, 1, 0, 0)        # group of 18 query heads
    assert lib.witcert_create(ctypes.byref(bad), ctypes.byref(h)) == _lib.EINVAL
    assert lib.witcert_gate(None, 0, 1.0, None) == _lib.EINVAL


def test_header_documents_each_entry_point():
    """Every declaration is directly preceded by a comment block."""
    lines = open(os.path.join(ROOT, "include", "witcert.h")).read().splitlines()
    for n in _declared():
        k = next(i for i, ln in enumerate(lines) if re.search(r"\b" + n + r"\s*\(", ln) and not ln.strip().startswith(("*", "/*")))
        prev = k - 1
        while prev >= 0 and not lines[prev].strip():
            prev -= 1
        assert lines[prev].strip().endswith("*/") or "/*" in lines[k], f"{n} has no comment"


def test_new_entry_points_reject_bad_arguments_without_the_gpu(lib_path):
    """Argument checks of the ragged, reset, paged and merge entry points come before any CUDA call."""
    import ctypes

    import kv_cache_quantization_witcert_gb300 as w
    from kv_cache_quantization_witcert_gb300 import _lib
    lib = w.load()
    h = ctypes.c_void_p()
    neg_pages = _lib.witcert_config(1, 4, 2, 128, 1, 16, 0, _lib.BF16, 0, 1, 0, 0, 0, 0, -1)
    assert lib.witcert_create(ctypes.byref(neg_pages), ctypes.byref(h)) == _lib.EINVAL
    paged_f32 = _lib.witcert_config(1, 4, 2, 128, 1, 16, 0, _lib.F32, 0, 1, 0, 0, 0, 0, 8)
    assert lib.witcert_create(ctypes.byref(paged_f32), ctypes.byref(h)) == _lib.EINVAL
    assert b"bf16" in lib.witcert_last_error()
    bad_scheme = _lib.witcert_config(1, 4, 2, 128, 1, 16, 9, _lib.BF16, 0, 1, 0, 0, 0, 0, 0)
    assert lib.witcert_create(ctypes.byref(bad_scheme), ctypes.byref(h)) == _lib.EINVAL
    counts = (ctypes.c_int32 * 1)(1)
    assert lib.witcert_write_ragged(None, 0, None, None, None, None, counts, None) == _lib.EINVAL
    assert lib.witcert_reset_sequence(None, 0, None) == _lib.EINVAL
    n = ctypes.c_int()
    assert lib.witcert_seq_length(None, 0, 0, ctypes.byref(n)) == _lib.EINVAL
    assert lib.witcert_write_hat(None, 0, None, None, None, None, 1, None) == _lib.EINVAL
    assert lib.witcert_merge_partials(None, 1, 1, 1, 0, None, None, None, None, None, None, None) == _lib.EINVAL
    fake = ctypes.c_void_p(1)
    assert lib.witcert_merge_partials(fake, 1, 1, 1, 7, fake, None, None, None, None, None, None) == _lib.EINVAL


def test_gate_shapes_and_fault_injection_are_checked_without_the_gpu(lib_path):
    """A gated cache whose sequences would hold more blocks than the gate ranks is refused at
    create; the selection call and the fault injection check their arguments first."""
    import ctypes

    import kv_cache_quantization_witcert_gb300 as w
    from kv_cache_quantization_witcert_gb300 import _lib
    lib = w.load()
    h = ctypes.c_void_p()
    too_long = _lib.witcert_config(1, 4, 2, 128, 1, 262144 + 16, 1, _lib.BF16, 0, 1, 0, 64, 0, 0, 0)
    assert lib.witcert_create(ctypes.byref(too_long), ctypes.byref(h)) == _lib.EINVAL
    assert b"gate" in lib.witcert_last_error()
    fake = ctypes.c_void_p(16)
    assert lib.witcert_gate_select(fake, None, 1, 4, 2, 16385, 1.0, fake, None) == _lib.EINVAL
    assert lib.witcert_gate_select(fake, None, 1, 3, 2, 16, 1.0, fake, None) == _lib.EINVAL
    assert lib.witcert_gate_select(fake, None, 1, 4, 2, 16, -1.0, fake, None) == _lib.EINVAL
    assert lib.witcert_gate_select(None, None, 1, 4, 2, 16, 1.0, fake, None) == _lib.EINVAL
    assert lib.witcert_inject_fault(None, _lib.FAULT_BACKING_LOST, 0) == _lib.EINVAL
