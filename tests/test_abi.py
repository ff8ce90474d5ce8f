"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/pkv.h declares.  Host-side argument validation is exercised with
invalid arguments only (it returns before any CUDA call), so no GPU is needed.
"""
import ctypes
import os
import re

import pytest

import paged_kv_attention_31_gb300 as pkv
from paged_kv_attention_31_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.lib()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("pkv_kv_append", "pkv_paged_attention", "pkv_paged_attention_workspace_size",
              "pkv_paged_prefill", "pkv_get_device_error", "pkv_status_string", "pkv_version",
              "pkv_copy_blocks", "pkv_cache_create", "pkv_cache_append", "pkv_cache_fork",
              "pkv_cache_preempt_for", "pkv_cache_block_tables"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} not exported"
    assert lib.pkv_version() == 101


def test_internal_symbols_hidden(lib):
    with pytest.raises(AttributeError):
        getattr(lib, "_ZN3pkv16launch_kv_appendERKNS_12AppendParamsEiP11CUstream_st")


def test_status_strings(lib):
    for s in range(8):
        assert pkv.status_string(s)
    assert pkv.status_string(99) == "unknown status"


def _desc(**kw):
    d = dict(num_blocks=8, num_kv_heads=2, block_size=16, head_dim=128, kv_dtype=0,
             k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return pkv.PoolDesc(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2), (dict(block_size=8), 2), (dict(kv_dtype=7), 1),
    (dict(num_blocks=0), 1), (dict(kv_dtype=1, k_scale=0.0), 1),
    (dict(kv_dtype=1, v_scale=float("nan")), 1)])
def test_pool_validation(lib, kw, status):
    d = _desc(**kw)
    z = ctypes.c_void_p(0)
    assert lib.pkv_kv_append(z, z, z, 4, z, z, ctypes.byref(d), z) == status


def test_argument_validation_before_any_cuda_call(lib):
    d = _desc()
    z = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(258)
    # null pointers
    assert lib.pkv_kv_append(z, z, z, 4, z, z, ctypes.byref(d), z) == 1
    # misaligned pool
    assert lib.pkv_kv_append(one, one, one, 4, odd, one, ctypes.byref(d), z) == 1
    assert lib.pkv_kv_append(z, z, z, 0, z, z, ctypes.byref(d), z) == 0  # no-op
    assert lib.pkv_kv_append(z, z, z, -1, z, z, ctypes.byref(d), z) == 1
    # group size 3 unsupported, Hq not a multiple of Hkv invalid
    args = lambda hq, part=0, ws=one: (one, one, one, ctypes.byref(d), one, 4, one, 2, hq, 100,
                                       0.1, part, ws, 1 << 20, one, z)
    assert lib.pkv_paged_attention(*args(6)) == 2
    assert lib.pkv_paged_attention(*args(3)) == 1
    assert lib.pkv_paged_attention(*args(4, part=24)) == 1     # not a multiple of block size
    assert lib.pkv_paged_attention(*args(4, ws=ctypes.c_void_p(272))) == 3  # misaligned workspace
    # prefill over an FP8 pool: the pool's scales are checked, and a group
    # size that does not divide 128 is not built
    d8 = _desc(kv_dtype=1, k_scale=0.0)
    assert lib.pkv_paged_prefill(one, one, one, one, ctypes.byref(d8), one, 4, one, 1, 4, 16, 16,
                                 0.1, one, z) == 1
    d8 = _desc(kv_dtype=1, k_scale=0.01, v_scale=0.02)
    assert lib.pkv_paged_prefill(one, one, one, one, ctypes.byref(d8), one, 4, one, 1, 6, 16, 16,
                                 0.1, one, z) == 2


def test_copy_blocks_validation_before_any_cuda_call(lib):
    d = _desc()
    z = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    assert lib.pkv_copy_blocks(one, one, ctypes.byref(d), one, 0, z) == 0      # no-op
    assert lib.pkv_copy_blocks(one, one, ctypes.byref(d), one, -1, z) == 1
    assert lib.pkv_copy_blocks(z, one, ctypes.byref(d), one, 2, z) == 1        # null pool
    assert lib.pkv_copy_blocks(one, one, ctypes.byref(d), z, 2, z) == 1        # null pairs
    assert lib.pkv_copy_blocks(one, ctypes.c_void_p(264), ctypes.byref(d), one, 2, z) == 1
    assert lib.pkv_copy_blocks(one, one, ctypes.byref(d), ctypes.c_void_p(258), 2, z) == 1


def test_fused_append_validation_before_any_cuda_call(lib):
    d = _desc()
    z = ctypes.c_void_p(0)
    one = ctypes.c_void_p(256)
    args = lambda T, kn=one, slots=one: (one, kn, one, slots, T, one, one, ctypes.byref(d), one, 4,
                                         one, 2, 8, 100, 0.1, 0, one, 1 << 20, one, z)
    assert lib.pkv_paged_attention_append(*args(-1)) == 1            # negative token count
    assert lib.pkv_paged_attention_append(*args(3, kn=z)) == 1       # null k_new
    assert lib.pkv_paged_attention_append(*args(3, slots=ctypes.c_void_p(260))) == 1  # misaligned
    bad = _desc(head_dim=96)
    assert lib.pkv_paged_attention_append(one, one, one, one, 3, one, one, ctypes.byref(bad), one,
                                          4, one, 2, 8, 100, 0.1, 0, one, 1 << 20, one, z) == 2


def test_workspace_size_is_positive(lib):
    d = _desc()
    assert lib.pkv_paged_attention_workspace_size(4, 8, 1000, 0, ctypes.byref(d)) > 0
    assert lib.pkv_paged_attention_workspace_size(4, 8, 1000, 24, ctypes.byref(d)) == 0


def test_self_test_validation_before_any_cuda_call(lib):
    out = ctypes.c_void_p(256)
    assert lib.pkv_self_test_bounded_wait(1000, None, None) == 1          # no output buffer
    assert lib.pkv_self_test_bounded_wait(0, out, None) == 1              # limit must be > 0
    assert lib.pkv_self_test_bounded_wait(3_000_000_000, out, None) == 1  # above the kernels' own
    assert lib.pkv_self_test_bounded_wait(1000, ctypes.c_void_p(258), None) == 1  # misaligned


@pytest.mark.parametrize("kw,nseq,status", [
    (None, 0, 1),                       # no pool descriptor, even with nothing to do
    (dict(head_dim=96), 4, 2), (dict(block_size=8), 4, 2), (dict(kv_dtype=7), 4, 1),
    (dict(num_blocks=0), 0, 1), (dict(), 0, 0),
    (dict(), -1, 1)])
def test_noalloc_reports_the_same_status_as_the_workspace_entry_point(lib, kw, nseq, status):
    # both decode entry points run the same host checks in the same order
    # (no CUDA call is reached for any of these arguments)
    z = ctypes.c_void_p(0)
    d = None if kw is None else _desc(**kw)
    dp = ctypes.byref(d) if d is not None else ctypes.POINTER(pkv.PoolDesc)()
    a = lib.pkv_paged_attention(z, z, z, dp, z, 4, z, nseq, 4, 64, 0.1, 0, z, 0, z, z)
    b = lib.pkv_paged_attention_noalloc(z, z, z, dp, z, 4, z, nseq, 4, 64, 0.1, 0, z, z)
    assert a == b == status
