"""Thin Python binding of libpkv.so, the GB300 paged-KV attention library.

Argument marshalling only: every step of the attention path runs in the CUDA
kernels behind the C ABI declared in include/pkv.h.  Tensors are torch CUDA
tensors; each call is enqueued on torch's current CUDA stream, or on the
`stream` argument when one is given (its default outputs and workspace are
then allocated on that stream).  There is no
CPU fallback: if the compiled library is missing, importing a function raises.

Functions mirror the C entry points:
    kv_append                       <- pkv_kv_append
    paged_attention_workspace_size  <- pkv_paged_attention_workspace_size
    paged_attention_plan            <- pkv_paged_attention_plan
    paged_attention                 <- pkv_paged_attention
    paged_attention_noalloc         <- pkv_paged_attention_noalloc
    paged_attention_append          <- pkv_paged_attention_append (append fused in)
    paged_prefill                   <- pkv_paged_prefill
    copy_blocks                     <- pkv_copy_blocks
    KVCacheManager                  <- pkv_cache_* (host page manager)
    get_device_error                <- pkv_get_device_error
    status_string                   <- pkv_status_string
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK = 0
PKV_ERR_DEVICE_BOUNDS = 5
PKV_ERR_DEVICE_TIMEOUT = 6
PKV_ERR_OUT_OF_BLOCKS = 7
KV_BF16 = 0
KV_FP8_E4M3 = 1

_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)} (status {status})"
        if status == 4:  # PKV_ERR_CUDA
            msg += f": {lib().pkv_last_cuda_error().decode()}"
        super().__init__(msg)


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("k_scales", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p)]


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m paged_kv_attention_31_gb300.build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_float, ctypes.c_size_t)
            pd = ctypes.POINTER(PoolDesc)
            L.pkv_kv_append.restype = i32
            L.pkv_kv_append.argtypes = [vp, vp, vp, i32, vp, vp, pd, vp]
            L.pkv_paged_attention_workspace_size.restype = sz
            L.pkv_paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, pd]
            L.pkv_paged_attention_plan.restype = i32
            L.pkv_paged_attention_plan.argtypes = [i32, i32, i32, i32, pd,
                                                   ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.pkv_paged_attention.restype = i32
            L.pkv_paged_attention.argtypes = [vp, vp, vp, pd, vp, i32, vp, i32, i32, i32, f32,
                                              i32, vp, sz, vp, vp]
            L.pkv_paged_attention_append.restype = i32
            L.pkv_paged_attention_append.argtypes = [vp, vp, vp, vp, i32, vp, vp, pd, vp, i32, vp,
                                                     i32, i32, i32, f32, i32, vp, sz, vp, vp]
            L.pkv_paged_attention_noalloc.restype = i32
            L.pkv_paged_attention_noalloc.argtypes = [vp, vp, vp, pd, vp, i32, vp, i32, i32, i32,
                                                      f32, i32, vp, vp]
            L.pkv_paged_attention_noalloc_max_scratch.restype = sz
            L.pkv_paged_attention_noalloc_max_scratch.argtypes = []
            L.pkv_paged_prefill.restype = i32
            L.pkv_paged_prefill.argtypes = [vp, vp, vp, vp, pd, vp, i32, vp, i32, i32, i32, i32,
                                            f32, vp, vp]
            L.pkv_copy_blocks.restype = i32
            L.pkv_copy_blocks.argtypes = [vp, vp, pd, vp, i32, vp]
            L.pkv_cache_create.restype = i32
            L.pkv_cache_create.argtypes = [i32, i32, i32, ctypes.POINTER(vp)]
            L.pkv_cache_destroy.restype = None
            L.pkv_cache_destroy.argtypes = [vp]
            for name in ("pkv_cache_num_free", "pkv_cache_num_seqs"):
                getattr(L, name).restype = i32
                getattr(L, name).argtypes = [vp]
            L.pkv_cache_length.restype = i32
            L.pkv_cache_length.argtypes = [vp, i64]
            L.pkv_cache_add.restype = i32
            L.pkv_cache_add.argtypes = [vp, i64]
            L.pkv_cache_fork.restype = i32
            L.pkv_cache_fork.argtypes = [vp, i64, i64, i32]
            L.pkv_cache_release.restype = i32
            L.pkv_cache_release.argtypes = [vp, i64]
            L.pkv_cache_blocks_needed.restype = i64
            L.pkv_cache_blocks_needed.argtypes = [vp, vp, vp, i32]
            L.pkv_cache_append.restype = i32
            L.pkv_cache_append.argtypes = [vp, vp, vp, i32, vp, i64, vp, i32,
                                           ctypes.POINTER(i64), ctypes.POINTER(i32)]
            L.pkv_cache_preempt_for.restype = i32
            L.pkv_cache_preempt_for.argtypes = [vp, i32, vp, i32, vp, i32, ctypes.POINTER(i32)]
            L.pkv_cache_block_tables.restype = i32
            L.pkv_cache_block_tables.argtypes = [vp, vp, i32, vp, vp]
            L.pkv_get_device_error.restype = i32
            L.pkv_get_device_error.argtypes = [ctypes.POINTER(i32), vp]
            L.pkv_self_test_bounded_wait.restype = i32
            L.pkv_self_test_bounded_wait.argtypes = [i64, vp, vp]
            L.pkv_last_cuda_error.restype = ctypes.c_char_p
            L.pkv_last_cuda_error.argtypes = []
            L.pkv_status_string.restype = ctypes.c_char_p
            L.pkv_status_string.argtypes = [i32]
            L.pkv_version.restype = i32
            L.pkv_version.argtypes = []
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != PKV_OK:
        raise PkvError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on(stream):
    """Context in which a call allocates its default tensors: the stream the
    call is enqueued on, so the caching allocator ties them to that stream
    and cannot hand their memory to another stream's allocation while the
    call's kernels still use it."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _is_fp8_pool(pool: torch.Tensor) -> bool:
    if pool.dtype in (torch.uint8, torch.float8_e4m3fn):
        return True
    if pool.dtype == torch.bfloat16:
        return False
    raise TypeError("pool must be bfloat16, uint8 or float8_e4m3fn")


def _scales_ptr(scales: Optional[torch.Tensor], hkv: int):
    if scales is None:
        return None
    if scales.dtype != torch.float32 or scales.numel() != hkv:
        raise ValueError("per-head scales must be float32 with one entry per kv head")
    return _ptr(scales).value


def pool_desc(k_pool: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0,
              k_scales: Optional[torch.Tensor] = None,
              v_scales: Optional[torch.Tensor] = None) -> PoolDesc:
    """Descriptor of a pool tensor [num_blocks, Hkv, block_size, head_dim].

    FP8 pools: per-tensor scales, or per-kv-head scale tensors (float32 [Hkv]
    on the device) that override them."""
    if k_pool.dim() != 4:
        raise ValueError("pool must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, P, D = k_pool.shape
    return PoolDesc(nb, hkv, P, D, KV_FP8_E4M3 if _is_fp8_pool(k_pool) else KV_BF16,
                    float(k_scale), float(v_scale), _scales_ptr(k_scales, hkv),
                    _scales_ptr(v_scales, hkv))


def _check_shapes(q, k_pool, v_pool, block_tables, context_lens, out, desc, rows):
    """The kernels see only pointers: q / out, both pools and the per-sequence
    tables must have the sizes the call implies (`rows` sequences)."""
    if v_pool.shape != k_pool.shape or v_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool and v_pool differ")
    if q.shape[2] != desc.head_dim:
        raise ValueError(f"q head_dim {q.shape[2]} differs from the pool's {desc.head_dim}")
    if out.shape != q.shape or out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16 with q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] < rows:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    if context_lens.dim() != 1 or context_lens.shape[0] < rows:
        raise ValueError("context_lens must hold one length per sequence")


def kv_append(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale=1.0, v_scale=1.0,
              stream=None, k_scales=None, v_scales=None) -> None:
    """Write new tokens' K/V rows ([T, Hkv, D] bf16) to their pool slots."""
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16:
        raise TypeError("k_new / v_new must be bfloat16")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    desc = pool_desc(k_pool, k_scale, v_scale, k_scales, v_scales)
    if v_pool.shape != k_pool.shape or v_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool and v_pool differ")
    T = int(slot_mapping.shape[0])
    if tuple(k_new.shape) != (T, desc.num_kv_heads, desc.head_dim) or k_new.shape != v_new.shape:
        raise ValueError("k_new / v_new must be [T, num_kv_heads, head_dim]")
    _check(lib().pkv_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(k_pool),
                               _ptr(v_pool), ctypes.byref(desc), _stream(stream)),
           "pkv_kv_append")


def paged_attention_workspace_size(num_seqs, num_q_heads, max_context_len, k_pool,
                                   partition_tokens=0, k_scale=1.0, v_scale=1.0) -> int:
    desc = pool_desc(k_pool, k_scale, v_scale)
    n = lib().pkv_paged_attention_workspace_size(int(num_seqs), int(num_q_heads),
                                                 int(max_context_len), int(partition_tokens),
                                                 ctypes.byref(desc))
    if n == 0:
        raise ValueError("invalid sizes for pkv_paged_attention_workspace_size")
    return int(n)


def paged_attention_plan(num_seqs, num_q_heads, max_context_len, k_pool, partition_tokens=0,
                         k_scale=1.0, v_scale=1.0):
    """(partition_tokens, max_splits) that paged_attention will use."""
    desc = pool_desc(k_pool, k_scale, v_scale)
    part, splits = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().pkv_paged_attention_plan(int(num_seqs), int(num_q_heads), int(max_context_len),
                                          int(partition_tokens), ctypes.byref(desc),
                                          ctypes.byref(part), ctypes.byref(splits)),
           "pkv_paged_attention_plan")
    return int(part.value), int(splits.value)


def paged_attention(q, k_pool, v_pool, block_tables, context_lens, max_context_len, scale,
                    out=None, workspace=None, k_scale=1.0, v_scale=1.0, partition_tokens=0,
                    stream=None, k_scales=None, v_scales=None) -> torch.Tensor:
    """Decode attention: q [B, Hq, D] bf16 -> out [B, Hq, D] bf16."""
    if q.dtype != torch.bfloat16 or q.dim() != 3:
        raise TypeError("q must be bfloat16 [num_seqs, num_q_heads, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables / context_lens must be int32")
    desc = pool_desc(k_pool, k_scale, v_scale, k_scales, v_scales)
    B, Hq, D = q.shape
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        _check_shapes(q, k_pool, v_pool, block_tables, context_lens, out, desc, B)
        if workspace is None:
            nbytes = paged_attention_workspace_size(B, Hq, max_context_len, k_pool,
                                                    partition_tokens, k_scale, v_scale)
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(lib().pkv_paged_attention(_ptr(q), _ptr(k_pool), _ptr(v_pool), ctypes.byref(desc),
                                     _ptr(block_tables), int(block_tables.shape[1]),
                                     _ptr(context_lens), int(B), int(Hq), int(max_context_len),
                                     float(scale), int(partition_tokens), _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()),
                                     _ptr(out), _stream(stream)),
           "pkv_paged_attention")
    return out


def paged_attention_append(q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables,
                           context_lens, max_context_len, scale, out=None, workspace=None,
                           k_scale=1.0, v_scale=1.0, partition_tokens=0, stream=None,
                           k_scales=None, v_scales=None) -> torch.Tensor:
    """kv_append + paged_attention in one call (the append runs in the
    attention's planning launch).  Returns out [B, Hq, D] bf16."""
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16:
        raise TypeError("k_new / v_new must be bfloat16")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if q.dtype != torch.bfloat16 or q.dim() != 3:
        raise TypeError("q must be bfloat16 [num_seqs, num_q_heads, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables / context_lens must be int32")
    desc = pool_desc(k_pool, k_scale, v_scale, k_scales, v_scales)
    if v_pool.shape != k_pool.shape or v_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool and v_pool differ")
    T = int(slot_mapping.shape[0])
    if tuple(k_new.shape) != (T, desc.num_kv_heads, desc.head_dim) or k_new.shape != v_new.shape:
        raise ValueError("k_new / v_new must be [T, num_kv_heads, head_dim]")
    B, Hq, D = q.shape
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        _check_shapes(q, k_pool, v_pool, block_tables, context_lens, out, desc, B)
        if workspace is None:
            nbytes = paged_attention_workspace_size(B, Hq, max_context_len, k_pool,
                                                    partition_tokens, k_scale, v_scale)
            workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    _check(lib().pkv_paged_attention_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(k_pool), _ptr(v_pool),
        ctypes.byref(desc), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens),
        B, Hq, int(max_context_len), float(scale), int(partition_tokens), _ptr(workspace),
        workspace.numel(), _ptr(out), _stream(stream)), "pkv_paged_attention_append")
    return out


def paged_attention_noalloc(q, k_pool, v_pool, block_tables, context_lens, max_context_len,
                            scale, out=None, k_scale=1.0, v_scale=1.0, partition_tokens=0,
                            stream=None, k_scales=None, v_scales=None) -> torch.Tensor:
    """Decode attention without a workspace, for callers that cannot allocate
    device scratch: the library's fixed device array is used instead (calls
    must not overlap on the GPU; the first call on a device does a one-time
    host set-up)."""
    if q.dtype != torch.bfloat16 or q.dim() != 3:
        raise TypeError("q must be bfloat16 [num_seqs, num_q_heads, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables / context_lens must be int32")
    desc = pool_desc(k_pool, k_scale, v_scale, k_scales, v_scales)
    B, Hq, D = q.shape
    if out is None:
        with _on(stream):
            out = torch.empty_like(q)
    _check_shapes(q, k_pool, v_pool, block_tables, context_lens, out, desc, B)
    _check(lib().pkv_paged_attention_noalloc(_ptr(q), _ptr(k_pool), _ptr(v_pool),
                                             ctypes.byref(desc), _ptr(block_tables),
                                             int(block_tables.shape[1]), _ptr(context_lens),
                                             int(B), int(Hq), int(max_context_len), float(scale),
                                             int(partition_tokens), _ptr(out), _stream(stream)),
           "pkv_paged_attention_noalloc")
    return out


def paged_prefill(q, cu_seqlens_q, k_pool, v_pool, block_tables, context_lens, max_q_len,
                  scale, out=None, stream=None, k_scale=1.0, v_scale=1.0, k_scales=None,
                  v_scales=None) -> torch.Tensor:
    """Causal chunked-prefill attention: q [T, Hq, D] bf16 -> out [T, Hq, D]
    bf16, over a bf16 or FP8 (E4M3, per-tensor or per-kv-head scales) pool."""
    if q.dtype != torch.bfloat16 or q.dim() != 3:
        raise TypeError("q must be bfloat16 [num_q_tokens, num_q_heads, head_dim]")
    for t in (cu_seqlens_q, block_tables, context_lens):
        if t.dtype != torch.int32:
            raise TypeError("cu_seqlens_q / block_tables / context_lens must be int32")
    desc = pool_desc(k_pool, k_scale, v_scale, k_scales, v_scales)
    T, Hq, D = q.shape
    n = int(context_lens.shape[0])
    if out is None:
        with _on(stream):
            out = torch.empty_like(q)
    _check_shapes(q, k_pool, v_pool, block_tables, context_lens, out, desc, n)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape[0] != n + 1:
        raise ValueError("cu_seqlens_q must be [num_seqs + 1]")
    _check(lib().pkv_paged_prefill(_ptr(q), _ptr(cu_seqlens_q), _ptr(k_pool), _ptr(v_pool),
                                   ctypes.byref(desc), _ptr(block_tables),
                                   int(block_tables.shape[1]), _ptr(context_lens), n, int(Hq),
                                   int(max_q_len), int(T), float(scale), _ptr(out),
                                   _stream(stream)),
           "pkv_paged_prefill")
    return out


def copy_blocks(k_pool, v_pool, pairs, stream=None, k_scale=1.0, v_scale=1.0) -> None:
    """Copy whole blocks of both pools: pairs is an int32 CUDA tensor [n, 2]
    of (source, destination) block ids, as KVCacheManager.append reports."""
    if pairs.dtype != torch.int32 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int32 [n, 2]")
    desc = pool_desc(k_pool, k_scale, v_scale)
    if v_pool.shape != k_pool.shape or v_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool and v_pool differ")
    n = int(pairs.shape[0])
    if n == 0:
        return
    _check(lib().pkv_copy_blocks(_ptr(k_pool), _ptr(v_pool), ctypes.byref(desc), _ptr(pairs),
                                 n, _stream(stream)), "pkv_copy_blocks")


def _np_ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


class KVCacheManager:
    """Host page manager of a paged KV pool (pkv_cache_* in the C library).

    Produces, in host numpy arrays, the device calls' inputs: slot mappings,
    copy-on-write block pairs, block tables and context lengths."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        h = ctypes.c_void_p(0)
        _check(lib().pkv_cache_create(int(num_blocks), int(block_size),
                                      int(max_blocks_per_seq), ctypes.byref(h)),
               "pkv_cache_create")
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.max_blocks_per_seq = int(max_blocks_per_seq)

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().pkv_cache_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may be gone already
            pass

    def num_free(self) -> int:
        return int(lib().pkv_cache_num_free(self._h))

    def num_seqs(self) -> int:
        return int(lib().pkv_cache_num_seqs(self._h))

    def length(self, seq_id: int) -> int:
        return int(lib().pkv_cache_length(self._h, int(seq_id)))

    def add(self, seq_id: int) -> int:
        return int(lib().pkv_cache_add(self._h, int(seq_id)))

    def fork(self, parent: int, child: int, num_tokens: int) -> int:
        return int(lib().pkv_cache_fork(self._h, int(parent), int(child), int(num_tokens)))

    def release(self, seq_id: int) -> int:
        return int(lib().pkv_cache_release(self._h, int(seq_id)))

    @staticmethod
    def _ids_counts(seq_ids, counts):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        if ids.shape != cnt.shape or ids.ndim != 1:
            raise ValueError("seq_ids and counts must be 1-D and of equal length")
        return ids, cnt

    def blocks_needed(self, seq_ids, counts) -> int:
        ids, cnt = self._ids_counts(seq_ids, counts)
        return int(lib().pkv_cache_blocks_needed(self._h, _np_ptr(ids), _np_ptr(cnt), len(ids)))

    def append(self, seq_ids, counts):
        """(status, slot_mapping int64 [sum counts], copies int32 [k, 2])."""
        ids, cnt = self._ids_counts(seq_ids, counts)
        n = len(ids)
        slots = np.empty(max(int(cnt[cnt > 0].sum()), 0), np.int64)
        copies = np.empty((max(n, 1), 2), np.int32)
        ns, nc = ctypes.c_int64(0), ctypes.c_int32(0)
        st = lib().pkv_cache_append(self._h, _np_ptr(ids), _np_ptr(cnt), n, _np_ptr(slots),
                                    slots.size, _np_ptr(copies), n, ctypes.byref(ns),
                                    ctypes.byref(nc))
        return int(st), slots[:ns.value].copy(), copies[:nc.value].copy()

    def preempt_for(self, needed: int, protected=()):
        """(status, list of released sequence ids, in release order)."""
        prot = np.ascontiguousarray(list(protected), dtype=np.int64)
        cap = max(self.num_seqs(), 1)
        victims = np.empty(cap, np.int64)
        nv = ctypes.c_int32(0)
        st = lib().pkv_cache_preempt_for(self._h, int(needed), _np_ptr(prot), len(prot),
                                         _np_ptr(victims), cap, ctypes.byref(nv))
        return int(st), [int(v) for v in victims[:nv.value]]

    def block_tables(self, seq_ids):
        """(int32 [n, max_blocks_per_seq] tables, int32 [n] context lengths)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = len(ids)
        tab = np.empty((n, self.max_blocks_per_seq), np.int32)
        lens = np.empty(n, np.int32)
        _check(lib().pkv_cache_block_tables(self._h, _np_ptr(ids), n, _np_ptr(tab),
                                            _np_ptr(lens)), "pkv_cache_block_tables")
        return tab, lens


def self_test_bounded_wait(limit_cycles: int = 1_000_000, stream=None) -> list:
    """Run the failure-path check (pkv_self_test_bounded_wait) and return its
    five results; the device error word then holds PKV_ERR_DEVICE_TIMEOUT."""
    # the buffer, the kernel and the read-back all on the call's stream: the
    # copy to the host waits for the kernel
    with _on(stream):
        out = torch.full((5,), -1, dtype=torch.int32, device="cuda")
        _check(lib().pkv_self_test_bounded_wait(int(limit_cycles), _ptr(out), _stream(stream)),
               "pkv_self_test_bounded_wait")
        return [int(x) for x in out.cpu()]


def get_device_error(stream=None) -> int:
    """Synchronise, then read and clear the device's sticky error word."""
    code = ctypes.c_int32(0)
    _check(lib().pkv_get_device_error(ctypes.byref(code), _stream(stream)),
           "pkv_get_device_error")
    return int(code.value)
