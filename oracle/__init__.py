"""Python marshalling for the fp64 C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg.  The product library never imports
or calls it, and it shares no code with the CUDA path.

All arrays are host numpy arrays: bf16 values as uint16 bit patterns, E4M3
values as uint8 codes, pools as [num_blocks, Hkv, P, D].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP8_E4M3 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (plain gcc, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            p, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                     ctypes.c_float, ctypes.c_double)
            L.pkvo_bf16_value.restype = f64
            L.pkvo_bf16_value.argtypes = [ctypes.c_uint16]
            L.pkvo_e4m3_value.restype = f64
            L.pkvo_e4m3_value.argtypes = [ctypes.c_uint8]
            L.pkvo_e4m3_encode.restype = ctypes.c_uint8
            L.pkvo_e4m3_encode.argtypes = [f32]
            L.pkvo_quantize_bf16.restype = ctypes.c_uint8
            L.pkvo_quantize_bf16.argtypes = [ctypes.c_uint16, f32]
            L.pkvo_e4m3_encode_array.restype = None
            L.pkvo_e4m3_encode_array.argtypes = [p, i64, p]
            L.pkvo_e4m3_value_array.restype = None
            L.pkvo_e4m3_value_array.argtypes = [p, i64, p]
            L.pkvo_kv_append.restype = i32
            L.pkvo_kv_append.argtypes = [p, p, p, i32, i32, i32, i32, i64, i32,
                                         f32, f32, p, p, p, p]
            L.pkvo_attention_one.restype = i32
            L.pkvo_attention_one.argtypes = [p, p, p, i32, f32, f32, i64, i32, i32,
                                             i32, i32, p, i32, f64, p]
            L.pkvo_paged_attention.restype = i32
            L.pkvo_paged_attention.argtypes = [p, p, p, i32, f32, f32, p, p, i64, i32, i32,
                                               i32, p, i32, p, i32, i32, f64, p]
            L.pkvo_paged_attention_rows.restype = i32
            L.pkvo_paged_attention_rows.argtypes = [p, p, p, i32, f32, f32, p, p, i64, i32,
                                                    i32, i32, p, i32, p, i32, p, p,
                                                    i32, f64, p]
            L.pkvo_paged_prefill.restype = i32
            L.pkvo_paged_prefill.argtypes = [p, p, p, p, i32, f32, f32, p, p, i64, i32, i32,
                                             i32, p, i32, p, i32, i32, f64, p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("array must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _scales(arr, hkv):
    """Optional per-kv-head scales -> (keepalive array, pointer or None)."""
    if arr is None:
        return None, None
    a = np.ascontiguousarray(arr, dtype=np.float32)
    if a.shape != (hkv,):
        raise ValueError("per-head scales must have one entry per kv head")
    return a, _ptr(a)


def _dtype_code(kv_dtype: str) -> int:
    return {"bf16": BF16, "fp8_e4m3": FP8_E4M3}[kv_dtype]


def _check_pool(pool: np.ndarray, kv_dtype: str):
    want = np.uint16 if kv_dtype == "bf16" else np.uint8
    if pool.dtype != want or pool.ndim != 4:
        raise TypeError(f"pool must be {want.__name__} [num_blocks, Hkv, P, D]")


# ---- element formats --------------------------------------------------------
def bf16_value(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    L = lib()
    return np.array([L.pkvo_bf16_value(int(b)) for b in bits.ravel()]).reshape(bits.shape)


def e4m3_value(codes) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib().pkvo_e4m3_value_array(_ptr(codes), codes.size, _ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().pkvo_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def quantize_bf16(bits: int, scale: float) -> int:
    return int(lib().pkvo_quantize_bf16(int(bits), float(scale)))


# ---- kv_append -------------------------------------------------------------
def kv_append(k_new, v_new, slot_mapping, k_pool, v_pool, kv_dtype="bf16",
              k_scale=1.0, v_scale=1.0, k_scales=None, v_scales=None) -> int:
    """Scatter new tokens into the pools in place; returns #out-of-pool slots.

    FP8: k_scales / v_scales (one per kv head) override k_scale / v_scale."""
    _check_pool(k_pool, kv_dtype)
    _check_pool(v_pool, kv_dtype)
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, hkv, P, D = k_pool.shape
    T = slots.shape[0]
    assert k_new.shape == (T, hkv, D) and v_new.shape == (T, hkv, D)
    ka, kptr = _scales(k_scales, hkv)
    va, vptr = _scales(v_scales, hkv)
    return lib().pkvo_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slots), T, hkv, P, D,
                                nb, _dtype_code(kv_dtype), k_scale, v_scale, kptr, vptr,
                                _ptr(k_pool), _ptr(v_pool))


# ---- attention ---------------------------------------------------------------
def copy_blocks(k_pool, v_pool, pairs) -> None:
    """Copy-on-write of shared blocks, in place: for each (source, destination)
    pair, the whole block (all kv heads) of both pools is duplicated.  The
    page's §4.1 / §4.2 ("TensorRT-LLM框架解析与高性能推理优化实践"): blocks are
    shared and reused, so a shared block is duplicated before an owner writes
    into it."""
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]


def paged_attention(q, k_pool, v_pool, block_tables, context_lens, scale,
                    kv_dtype="bf16", k_scale=1.0, v_scale=1.0, k_scales=None,
                    v_scales=None) -> np.ndarray:
    """fp64 out [B, Hq, D] for every (sequence, q head)."""
    _check_pool(k_pool, kv_dtype)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    nb, hkv, P, D = k_pool.shape
    B, Hq, Dq = q.shape
    assert Dq == D and Hq % hkv == 0 and bt.shape[0] == B and cl.shape == (B,)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    ka, kptr = _scales(k_scales, hkv)
    va, vptr = _scales(v_scales, hkv)
    bad = lib().pkvo_paged_attention(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                     _dtype_code(kv_dtype), k_scale, v_scale, kptr, vptr,
                                     nb, hkv,
                                     P, D, _ptr(bt), bt.shape[1], _ptr(cl), B, Hq,
                                     float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} rows reference pages outside the pool")
    return out


def paged_attention_rows(q, k_pool, v_pool, block_tables, context_lens, scale,
                         seq_ids, head_ids, kv_dtype="bf16", k_scale=1.0,
                         v_scale=1.0, k_scales=None, v_scales=None) -> np.ndarray:
    """fp64 out [n, D] for the listed (sequence, q head) pairs."""
    _check_pool(k_pool, kv_dtype)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    si = np.ascontiguousarray(seq_ids, dtype=np.int32)
    hi = np.ascontiguousarray(head_ids, dtype=np.int32)
    nb, hkv, P, D = k_pool.shape
    Hq = q.shape[1]
    out = np.zeros((si.shape[0], D), dtype=np.float64)
    ka, kptr = _scales(k_scales, hkv)
    va, vptr = _scales(v_scales, hkv)
    bad = lib().pkvo_paged_attention_rows(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                          _dtype_code(kv_dtype), k_scale, v_scale, kptr,
                                          vptr, nb,
                                          hkv, P, D, _ptr(bt), bt.shape[1], _ptr(cl),
                                          Hq, _ptr(si), _ptr(hi), si.shape[0],
                                          float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} rows reference pages outside the pool")
    return out


def paged_prefill(q, cu_seqlens_q, k_pool, v_pool, block_tables, context_lens,
                  scale, kv_dtype="bf16", k_scale=1.0, v_scale=1.0, k_scales=None,
                  v_scales=None) -> np.ndarray:
    """fp64 out [T_p, Hq, D]: causal attention of packed chunk tokens (FP8
    pools: per-tensor scales, or per-kv-head k_scales / v_scales)."""
    _check_pool(k_pool, kv_dtype)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    nb, hkv, P, D = k_pool.shape
    T, Hq, _ = q.shape
    n = cl.shape[0]
    assert cu.shape == (n + 1,) and int(cu[-1]) == T
    out = np.zeros((T, Hq, D), dtype=np.float64)
    ka, kptr = _scales(k_scales, hkv)
    va, vptr = _scales(v_scales, hkv)
    bad = lib().pkvo_paged_prefill(_ptr(q), _ptr(cu), _ptr(k_pool), _ptr(v_pool),
                                   _dtype_code(kv_dtype), k_scale, v_scale, kptr, vptr, nb,
                                   hkv, P, D, _ptr(bt), bt.shape[1], _ptr(cl), n, Hq,
                                   float(scale), _ptr(out))
    if bad:
        raise ValueError(f"{bad} rows reference pages outside the pool")
    return out
