"""The C ABI library loads and exports every symbol include/nt.h declares; host-side argument
validation answers without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from packed_weight_gemv_gb300 import build as nt_build
from packed_weight_gemv_gb300 import nt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nt_build.build()
    return nt.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nt_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(nt.EXPORTS)


def test_abi_version_and_status_strings(lib):
    assert lib.nt_abi_version() == 1
    for s in range(8):
        assert lib.nt_status_string(s)
    assert b"unknown" in lib.nt_status_string(99)


def test_size_queries(lib):
    assert nt.nt_repack_size(1536, 512) == 1536 * 512 // 4
    assert nt.nt_repack_size(5, 16) == 8 * 512 // 4
    assert nt.nt_repack_size(4096, 12288) == 4096 * 12288 // 4
    assert nt.nt_int8_logits_workspace_size(151936, 4096, 1) > 0
    with pytest.raises(nt.NtError) as e:
        nt.nt_repack_size(4, 15)
    assert e.value.status == nt.NT_ERR_INVALID_ARG


def _gemv(lib, w, layout, N, K, q, y, B=1):
    vp = ctypes.c_void_p
    return lib.nt_ternary_gemm(vp(w), layout, vp(0x1000), N, K, vp(q), vp(0x2000), B, vp(y),
                               None, None, 0, None)


def test_argument_errors_without_gpu(lib):
    # Validation happens before any device call, so these answer on a machine with no GPU.
    assert _gemv(lib, 0x10000, 1, 16, 15, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10000, 1, 0, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10000, 7, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    assert _gemv(lib, 0x10008, 1, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_ALIGNMENT
    assert _gemv(lib, 0x10000, 1, 16, 16, 0x20004, 0x30000) == nt.NT_ERR_ALIGNMENT
    assert _gemv(lib, 0, 1, 16, 16, 0x20000, 0x30000) == nt.NT_ERR_INVALID_ARG
    # the tensor-core path (tiled, B >= 64) needs a workspace: refused before any device call
    assert _gemv(lib, 0x10000, 1, 256, 512, 0x20000, 0x30000, B=64) == nt.NT_ERR_WORKSPACE
    # every workspace starts with the 256-byte status header (16 bytes used, the rest keeps the
    # data's alignment)
    H = 256
    # prefill: the status header and an f16 copy of the activations (the weights stay packed)
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 64, nt.NT_LAYOUT_TILED) == H + 64 * 512 * 2
    # 2..16 vectors, from 128 rows: an optional workspace of e4m3 digit rows (16 for B <= 8,
    # else 32, K rounded up to 128), int32 partial sums [B][N] and one counter per 128-row
    # tile, rounded up to 16 bytes; below 128 rows sums and one counter per 256 rows; none for
    # one vector or above 16
    r16 = lambda b: (b + 15) // 16 * 16  # noqa: E731
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 16, nt.NT_LAYOUT_TILED) == H + r16(32 * 512 + 16 * 256 * 4 + 2 * 4)
    assert nt.nt_ternary_gemm_workspace_size(1000, 512, 3, nt.NT_LAYOUT_TILED) == H + r16(16 * 512 + 3 * 1000 * 4 + 8 * 4)
    assert nt.nt_ternary_gemm_workspace_size(1000, 208, 3, nt.NT_LAYOUT_TILED) == H + r16(16 * 256 + 3 * 1000 * 4 + 8 * 4)
    assert nt.nt_ternary_gemm_workspace_size(100, 512, 3, nt.NT_LAYOUT_TILED) == H + (3 * 100 * 4 + 4 + 15) // 16 * 16
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 1, nt.NT_LAYOUT_TILED) == 0
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 17, nt.NT_LAYOUT_TILED) == 0
    assert nt.nt_ternary_gemm_workspace_size(256, 512, 16, nt.NT_LAYOUT_PLAIN) == 0
    assert b"multiple of 16" in lib.nt_last_error_string() or True
    vp = ctypes.c_void_p
    assert lib.nt_quantize_act(None, 1, 16, vp(0x100), vp(0x200), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_quantize_act(vp(0x102), 1, 16, vp(0x100), vp(0x200), None) == nt.NT_ERR_ALIGNMENT
    r = lib.nt_int8_logits_argmax(vp(0x1000), vp(0x2000), 10, 16, vp(0x3000), vp(0x4000), 1,
                                  None, vp(0x5000), None, 0, None)
    assert r == nt.NT_ERR_WORKSPACE
    r = lib.nt_int8_logits_argmax(vp(0x1008), vp(0x2000), 10, 16, vp(0x3000), vp(0x4000), 1,
                                  None, vp(0x5000), vp(0x6000), 1 << 20, None)
    assert r == nt.NT_ERR_ALIGNMENT


def test_validate_argument_errors_without_gpu(lib):
    vp, n = ctypes.c_void_p, ctypes.c_uint64(0)
    assert lib.nt_validate_ternary(None, 4, 16, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1000), 4, 15, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1000), 0, 16, ctypes.byref(n), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_validate_ternary(vp(0x1002), 4, 16, ctypes.byref(n), None) == nt.NT_ERR_ALIGNMENT
    assert b"10" in lib.nt_status_string(nt.NT_ERR_INVALID_CODE)


def test_status_and_fault_hook_without_gpu(lib):
    st = ctypes.c_int(-1)
    assert lib.nt_workspace_status(None, ctypes.byref(st)) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_workspace_status(ctypes.c_void_p(0x1000), None) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(4, 1.0) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(-1, 1.0) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_set_test_fault(0, 0.0) == nt.NT_OK
    assert lib.nt_decode_plan_capture_size(None, ctypes.byref(ctypes.c_size_t(0))) == nt.NT_ERR_INVALID_ARG
    assert lib.nt_decode_plan_set_capture(None, None) == nt.NT_ERR_INVALID_ARG


def test_plan_descriptor_errors_without_gpu(lib):
    d = nt.nt_decode_desc()
    h = ctypes.c_void_p(None)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    arr = (nt.nt_proj * 7)()
    for i in range(7):
        arr[i] = nt.nt_proj(64, 48, 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000)
    d.n_layers, d.batch, d.proj = 1, 17, ctypes.cast(arr, ctypes.POINTER(nt.nt_proj))
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    d.batch, d.mode = 1, 5
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    d.mode = 0
    arr[3] = nt.nt_proj(64, 40, 0x10000, 0x20000, None, 0x30000, 0x40000, 0x50000)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_INVALID_ARG
    arr[3] = nt.nt_proj(64, 48, 0x10004, 0x20000, None, 0x30000, 0x40000, 0x50000)
    assert lib.nt_decode_plan_create(ctypes.byref(d), ctypes.byref(h)) == nt.NT_ERR_ALIGNMENT
    assert not h.value
