"""The C-ABI library: it loads, exports every entry point its header declares,
and rejects bad host-side arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from speculative_verify_accept_step_b300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "idlm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idlm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_verify_accept_step_b300.build import build
    build()
    return _lib.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("idlm_isd_attention", "idlm_isd_accept", "idlm_kv_commit",
              "idlm_isd_attention_workspace_size", "idlm_isd_accept_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.idlm_status_string(0) == b"ok"
    assert lib.idlm_status_string(3) == b"workspace missing or too small"
    assert lib.idlm_version() >= 100


def test_null_pointers_are_rejected_without_a_gpu(lib):
    vp = ctypes.c_void_p
    rc = lib.idlm_isd_attention(*([None] * 6), 1, None, None, 1, 3, 4, 1, 64, 16, 1, 3,
                                0.125, 0, None, None, 0, None, None)
    assert rc == 1
    rc = lib.idlm_kv_commit(None, None, None, 1, None, None, None, None, None, None, 1, 3, 1, 64,
                            16, 1, 0, None, None, None)
    assert rc == 1
    args = [None, 1, 1024] + [None] * 5 + [1, None] + [1, 3, 2, 1.0, 0, 0, 0] + [None] * 10 + [None, 0, None, None]
    assert lib.idlm_isd_accept(*args) == 1
    del vp


def test_bad_sizes_are_rejected_without_a_gpu(lib):
    dummy = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    p = [dummy] * 6
    # Hq not a multiple of Hkv
    rc = lib.idlm_isd_attention(*p, 4, dummy, dummy, 1, 3, 6, 4, 64, 16, 8, 3, 0.125, 0,
                                dummy, dummy, 1 << 20, dummy, None)
    assert rc == 1
    # accept: N = 1 is not a stride
    args = [dummy, 1, 1024] + [dummy] * 5 + [4, dummy] + [1, 3, 1, 1.0, 0, 0, 0] + [dummy] * 10 + [dummy, 1 << 20, dummy, None]
    assert lib.idlm_isd_accept(*args) == 1
    # accept: V not a multiple of 8
    args = [dummy, 1, 1020] + [dummy] * 5 + [4, dummy] + [1, 3, 2, 1.0, 0, 0, 0] + [dummy] * 10 + [dummy, 1 << 20, dummy, None]
    assert lib.idlm_isd_accept(*args) == 2
    # accept: workspace too small
    args = [dummy, 1, 1024] + [dummy] * 5 + [4, dummy] + [1, 3, 2, 1.0, 0, 0, 0] + [dummy] * 10 + [dummy, 8, dummy, None]
    assert lib.idlm_isd_accept(*args) == 3
    # commit: fp32 row of 3 floats is not a 16-byte multiple
    rc = lib.idlm_kv_commit(dummy, dummy, dummy, 1, dummy, dummy, dummy, dummy, dummy, dummy,
                            1, 3, 1, 3, 16, 1, 0, None, dummy, None)
    assert rc == 2


def test_gated_lora_host_checks_without_a_gpu(lib):
    """idlm_gated_lora validates its arguments on the host, before any CUDA call."""
    d = ctypes.c_void_p(256)      # 256-byte aligned, never dereferenced
    odd = ctypes.c_void_p(264)    # 8-byte aligned only
    ws = lib.idlm_gated_lora_workspace_size(448, 4096, 1024, 16)
    assert ws > 0
    # null pointers (the adapter's may be null only at rank 0)
    assert lib.idlm_gated_lora(None, d, d, d, d, 1.0, 448, 4096, 1024, 16, d, d, ws, d, None) == 1
    assert lib.idlm_gated_lora(d, d, None, d, d, 1.0, 448, 4096, 1024, 16, d, d, ws, d, None) == 1
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4096, 1024, 16, d, d, ws, None, None) == 1
    # sizes: M = 0, K not a multiple of 8, r not a multiple of 8 or above 128
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 0, 4096, 1024, 16, d, d, ws, d, None) == 1
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4092, 1024, 16, d, d, ws, d, None) == 2
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4096, 1024, 12, d, d, ws, d, None) == 2
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4096, 1024, 136, d, d, ws, d, None) == 2
    # operands must be 16-byte aligned (TMA)
    assert lib.idlm_gated_lora(odd, d, d, d, d, 1.0, 448, 4096, 1024, 16, d, d, ws, d, None) == 1
    # workspace: too small, or not 256-byte aligned
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4096, 1024, 16, d, d, ws - 1, d, None) == 3
    assert lib.idlm_gated_lora(d, d, d, d, d, 1.0, 448, 4096, 1024, 16, d, odd, ws, d, None) == 3


def test_gated_lora_workspace_size(lib):
    f = lib.idlm_gated_lora_workspace_size
    assert f(0, 4096, 1024, 16) == 0 and f(448, 4096, 1024, -1) == 0
    # rank 0 (no adapter) is a plain projection: partial tiles only
    assert 0 < f(448, 4096, 1024, 0) < f(448, 4096, 1024, 16)
    # grows with N (the padded B rows) and with the rank (the adapter operands)
    assert f(448, 4096, 2048, 16) > f(448, 4096, 1024, 16)
    assert f(448, 4096, 1024, 72) > f(448, 4096, 1024, 16)
    g = lib.idlm_gated_lora_grouped_workspace_size
    assert g(448, 4096, 6144, 16, 1) == f(448, 4096, 6144, 16)
    assert g(448, 4096, 6144, 16, 3) > g(448, 4096, 6144, 16, 1)
    # token rows beyond one 448-row slice reuse the slice's workspace
    assert f(4480, 4096, 1024, 16) == f(448, 4096, 1024, 16)


def test_grouped_gated_lora_host_checks_without_a_gpu(lib):
    d = ctypes.c_void_p(256)
    ws = lib.idlm_gated_lora_grouped_workspace_size(448, 4096, 6144, 16, 3)
    rows = (ctypes.c_int * 3)(4096, 1024, 1024)
    bad_sum = (ctypes.c_int * 3)(4096, 1024, 1000)
    unaligned = (ctypes.c_int * 3)(4000, 1120, 1024)
    f = lib.idlm_gated_lora_grouped
    assert f(d, d, d, d, d, 1.0, 448, 4096, 6144, 16, 3, None, d, d, ws, d, None) == 1
    assert f(d, d, d, d, d, 1.0, 448, 4096, 6144, 16, 3, bad_sum, d, d, ws, d, None) == 1
    assert f(d, d, d, d, d, 1.0, 448, 4096, 6144, 16, 3, unaligned, d, d, ws, d, None) == 2
    assert f(d, d, d, d, d, 1.0, 448, 4096, 6144, 16, 5, rows, d, d, ws, d, None) == 2
    assert f(d, d, d, d, d, 1.0, 448, 4096, 6144, 16, 3, rows, d, d, ws - 1, d, None) == 3
