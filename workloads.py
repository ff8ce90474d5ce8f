"""Seeded synthetic inputs for one paged-KV attention step.

This module builds inputs only: sequence lengths, page allocation and block
tables, slot mappings, and the values of q, K and V.  It holds none of the
attention arithmetic (no gather, no softmax, no FP8 encoding, no rounding of
results), so both the CPU oracle and the CUDA library can consume it without
sharing any of the method's code.

Values.  Every value is a pure function of (seed, stream, linear index): a
counter-based integer hash turns the index into eight 16-bit uniforms whose
sum, centred and scaled to unit variance, approximates N(0, 1) (Irwin-Hall
with n = 8; |x| < 4.9).  The hash uses only integer xor/shift/multiply on
values below 2^63 plus one fp32 multiply and an RNE cast to bf16, so the same
bits come out on the CPU and on the GPU.  That lets a GPU test fill a
multi-GB pool on the device while the oracle regenerates, on the host, only
the pages of the sequences it checks.

Shapes follow the in-flight-batching decode step of the TensorRT-LLM pages
("KV缓存管理细节", §4.2: paged KV, non-contiguous physical pages; §6.2 Paged
Attention: block_tables [num_seqs, max_blocks]); prefix pages shared between
sequences follow the shared-prefix item of §6.2; chunked context follows §5.3.
Pool layout: k_pool, v_pool = [num_blocks, num_kv_heads, block_size, head_dim].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# ----------------------------------------------------------------------------
# counter-based value generator
# ----------------------------------------------------------------------------
_M32 = 0xFFFFFFFF
_STREAMS = {"k": 1, "v": 2, "q": 3, "k_new": 4, "v_new": 5, "q_prefill": 6,
            "aux": 7}
# fp32 constant: sqrt(12 / 8) / 65536 maps a centred sum of eight 16-bit
# uniforms to unit variance.
_UNIT = float(np.float32(math.sqrt(1.5) / 65536.0))
# Largest magnitude the generator can produce (before the bf16 cast).
VALUE_BOUND = float(np.float32(np.float32(262148.0) * np.float32(_UNIT)))
# Per-tensor FP8 scales used by the FP8 workloads: the value bound maps to the
# largest finite E4M3 magnitude (448), so no generated value saturates.
FP8_SCALE = float(np.float32(VALUE_BOUND / 448.0))


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit avalanche hash on an int64 tensor holding values in [0, 2^32).

    Multipliers are below 2^31, so no intermediate leaves [0, 2^63).
    """
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & _M32
    x = x ^ (x >> 15)
    x = (x * 0x68E31DA5) & _M32
    x = x ^ (x >> 16)
    return x


def _mix32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x68E31DA5) & _M32
    x ^= x >> 16
    return x


def normal_bf16(seed: int, stream: str, index: torch.Tensor) -> torch.Tensor:
    """Approximately N(0,1) bf16 values for int64 linear indices ``index``."""
    if index.dtype != torch.int64:
        raise TypeError("index must be int64")
    sid = _STREAMS[stream]
    base = _mix32_int(seed * 0x9E3779B1 + sid * 0x85EBCA77 + 0x165667B1)
    base_hi = _mix32_int(base ^ 0x27D4EB2F)
    lo = index & _M32
    hi = index >> 32
    h = _mix32(lo ^ base)
    h = _mix32(h ^ _mix32((hi + base_hi) & _M32))
    total = None
    for c in (0x3C6EF372, 0xA54FF53A, 0x510E527F, 0x1F83D9AB):
        w = _mix32(h ^ c)
        part = (w & 0xFFFF) + (w >> 16)
        total = part if total is None else total + part
        del w, part
    # sum of eight (u + 0.5) / 65536 minus its mean 4, in units of 1/65536
    centred = (total + 4 - 262144).to(torch.float32)
    del total, h, lo, hi
    vals = centred * torch.tensor(_UNIT, dtype=torch.float32, device=index.device)
    return vals.to(torch.bfloat16)


def pool_values(seed: int, which: str, page_ids, num_kv_heads: int,
                block_size: int, head_dim: int, device="cpu") -> torch.Tensor:
    """bf16 [len(page_ids), Hkv, P, D]: generator values of pool pages.

    Element (page, h, o, d) has linear index ((page*Hkv + h)*P + o)*D + d, the
    row-major index of that element in the whole pool.
    """
    pages = torch.as_tensor(np.asarray(page_ids, dtype=np.int64), device=device)
    per_page = num_kv_heads * block_size * head_dim
    inner = torch.arange(per_page, dtype=torch.int64, device=device)
    idx = pages[:, None] * per_page + inner[None, :]
    out = normal_bf16(seed, which, idx.reshape(-1))
    return out.reshape(len(pages), num_kv_heads, block_size, head_dim)


def pool_values_head(seed: int, which: str, page_ids, head: int, num_kv_heads: int,
                     block_size: int, head_dim: int, device="cpu") -> torch.Tensor:
    """bf16 [len(page_ids), P, D]: the kv-head ``head`` slice of pool pages."""
    pages = torch.as_tensor(np.asarray(page_ids, dtype=np.int64), device=device)
    run = block_size * head_dim
    inner = torch.arange(run, dtype=torch.int64, device=device)
    idx = (pages[:, None] * num_kv_heads + head) * run + inner[None, :]
    out = normal_bf16(seed, which, idx.reshape(-1))
    return out.reshape(len(pages), block_size, head_dim)


def fill_pool_(pool: torch.Tensor, seed: int, which: str,
               pages_per_chunk: int = 0) -> torch.Tensor:
    """Fill a bf16 pool [num_blocks, Hkv, P, D] in place, chunk by chunk."""
    nb, hkv, p, d = pool.shape
    if pages_per_chunk <= 0:
        pages_per_chunk = max(1, (1 << 26) // (hkv * p * d))
    for start in range(0, nb, pages_per_chunk):
        stop = min(nb, start + pages_per_chunk)
        ids = np.arange(start, stop, dtype=np.int64)
        pool[start:stop] = pool_values(seed, which, ids, hkv, p, d,
                                       device=pool.device)
    return pool


def dense_values(seed: int, stream: str, shape, device="cpu") -> torch.Tensor:
    """bf16 tensor of ``shape`` whose element i (row-major) is value i."""
    n = int(np.prod(shape))
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return normal_bf16(seed, stream, idx).reshape(tuple(shape))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of a bf16 tensor (raw bits)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    """One mixed batch: decode sequences and (optionally) prefill chunks.

    context lengths INCLUDE the tokens appended in this step (the new decode
    token, or the whole prefill chunk): the step appends first, then attends.
    Block-table entries past a sequence's last page are -1.
    """
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str                     # "bf16" | "fp8_e4m3"
    num_blocks: int
    context_lens: np.ndarray          # int32 [B] decode sequences
    block_tables: np.ndarray          # int32 [B, max_blocks]
    prefill_context_lens: np.ndarray  # int32 [n] prefill sequences
    prefill_chunk_lens: np.ndarray    # int32 [n]
    prefill_block_tables: np.ndarray  # int32 [n, max_blocks]
    k_scale: float = 1.0
    v_scale: float = 1.0
    shared_prefix_tokens: int = 0
    num_sharers: int = 0
    k_scales: Optional[np.ndarray] = None  # float32 [Hkv]: per-kv-head FP8 scales
    v_scales: Optional[np.ndarray] = None  # (override k_scale / v_scale when set)

    def head_scales(self, h: int):
        """(k scale, v scale) that apply to kv head h."""
        ks = self.k_scale if self.k_scales is None else float(self.k_scales[h])
        vs = self.v_scale if self.v_scales is None else float(self.v_scales[h])
        return ks, vs

    def scale_tensors(self, device="cpu"):
        """Per-head scale arrays as float32 tensors, or (None, None)."""
        if self.k_scales is None:
            return None, None
        return (torch.from_numpy(np.asarray(self.k_scales, np.float32)).to(device),
                torch.from_numpy(np.asarray(self.v_scales, np.float32)).to(device))

    # -- derived sizes ------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_prefill(self) -> int:
        return int(self.prefill_context_lens.shape[0])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8_e4m3" else 2

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def num_prefill_tokens(self) -> int:
        return int(self.prefill_chunk_lens.sum()) if self.num_prefill else 0

    def cu_seqlens_q(self) -> np.ndarray:
        cu = np.zeros(self.num_prefill + 1, dtype=np.int32)
        if self.num_prefill:
            cu[1:] = np.cumsum(self.prefill_chunk_lens)
        return cu

    # -- where the step's new tokens go -------------------------------------
    def decode_slot_mapping(self) -> np.ndarray:
        """int64 [B]: pool slot (page*P + offset) of each decode token.

        A sequence of length 0 appends nothing: its slot is -1 (skipped)."""
        pos = self.context_lens.astype(np.int64) - 1
        rows = np.arange(self.num_seqs)
        page = self.block_tables[rows, np.maximum(pos, 0) // self.block_size].astype(np.int64)
        slot = page * self.block_size + np.maximum(pos, 0) % self.block_size
        return np.where(pos >= 0, slot, -1)

    def prefill_slot_mapping(self) -> np.ndarray:
        """int64 [T_p]: pool slots of the prefill chunk tokens, packed."""
        out = []
        for s in range(self.num_prefill):
            L = int(self.prefill_context_lens[s])
            C = int(self.prefill_chunk_lens[s])
            pos = np.arange(L - C, L, dtype=np.int64)
            page = self.prefill_block_tables[s, pos // self.block_size]
            out.append(page.astype(np.int64) * self.block_size + pos % self.block_size)
        if not out:
            return np.zeros(0, dtype=np.int64)
        return np.concatenate(out)

    def append_slot_mapping(self) -> np.ndarray:
        """Slots of all tokens appended this step: decode tokens first."""
        return np.concatenate([self.decode_slot_mapping(),
                               self.prefill_slot_mapping()])

    @property
    def num_append_tokens(self) -> int:
        return self.num_seqs + self.num_prefill_tokens

    # -- value tensors ------------------------------------------------------
    def q_decode(self, device="cpu") -> torch.Tensor:
        return dense_values(self.seed, "q",
                            (self.num_seqs, self.num_q_heads, self.head_dim), device)

    def q_prefill(self, device="cpu") -> torch.Tensor:
        return dense_values(self.seed, "q_prefill",
                            (self.num_prefill_tokens, self.num_q_heads,
                             self.head_dim), device)

    def kv_new(self, device="cpu"):
        """bf16 k_new, v_new [T, Hkv, D] for every appended token."""
        shape = (self.num_append_tokens, self.num_kv_heads, self.head_dim)
        return (dense_values(self.seed, "k_new", shape, device),
                dense_values(self.seed, "v_new", shape, device))

    def pool_source(self, which: str, page_ids, device="cpu") -> torch.Tensor:
        """bf16 source values of the given pool pages (before any append)."""
        return pool_values(self.seed, which, page_ids, self.num_kv_heads,
                           self.block_size, self.head_dim, device)

    # -- algorithmic byte counts -------------------------------------------
    def decode_kv_bytes(self, unique: bool = True) -> int:
        """K+V bytes the decode attention must read.

        With ``unique``, pages shared by prefix reuse count once.
        """
        per_tok = self.num_kv_heads * 2 * self.head_dim * self.elem_bytes
        toks = int(self.context_lens.astype(np.int64).sum())
        if unique and self.num_sharers > 1:
            toks -= (self.num_sharers - 1) * self.shared_prefix_tokens
        return toks * per_tok

    def prefill_flops(self) -> int:
        """Causal-exact flops of the prefill attention (QK^T and PV, 2 flops
        per multiply-add): chunk token i of sequence s sees L - C + i + 1 keys."""
        total = 0
        for s in range(self.num_prefill):
            L, C = int(self.prefill_context_lens[s]), int(self.prefill_chunk_lens[s])
            keys = C * (L - C) + C * (C + 1) // 2
            total += keys * self.num_q_heads * 4 * self.head_dim
        return total

    def decode_step_bytes(self, unique: bool = True) -> int:
        """Algorithmic bytes of one decode step (append + attention)."""
        B, Hq, Hkv, D = self.num_seqs, self.num_q_heads, self.num_kv_heads, self.head_dim
        kv = self.decode_kv_bytes(unique)
        q_out = 2 * B * Hq * D * 2                       # q in, out, both bf16
        pages = int(np.sum((self.context_lens.astype(np.int64) + self.block_size - 1)
                           // self.block_size))
        tables = pages * 4 + B * 4                        # block-table entries + lens
        append = B * (8 + Hkv * D * 2 * 2 + Hkv * D * 2 * self.elem_bytes)
        return kv + q_out + tables + append


def _pages(n_tokens: np.ndarray, P: int) -> np.ndarray:
    return (n_tokens.astype(np.int64) + P - 1) // P


def _allocate(rng, lens: np.ndarray, P: int, max_blocks: int,
              shared_tokens: int = 0, num_sharers: int = 0,
              num_blocks: Optional[int] = None, pool_factor: float = 1.25):
    """Block tables over a randomly permuted pool.

    Sequences 0..num_sharers-1 share the first shared_tokens/P pages.
    """
    n = len(lens)
    need = _pages(lens, P)
    sp = shared_tokens // P if num_sharers > 0 else 0
    own = need.copy()
    own[:num_sharers] -= sp
    unique = int(own.sum()) + sp
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * unique))
    if unique > num_blocks:
        raise ValueError("pool too small")
    ids = rng.permutation(num_blocks).astype(np.int32)
    tables = np.full((n, max_blocks), -1, dtype=np.int32)
    cursor = 0
    shared_ids = ids[cursor:cursor + sp]
    cursor += sp
    for s in range(n):
        first = 0
        if s < num_sharers:
            tables[s, :sp] = shared_ids
            first = sp
        k = int(need[s]) - first
        tables[s, first:first + k] = ids[cursor:cursor + k]
        cursor += k
    return tables, num_blocks


def _uniform_int(rng, lo, hi, n):
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


def _log_uniform_int(rng, lo, hi, n):
    x = np.exp(rng.uniform(math.log(lo), math.log(hi + 1), size=n))
    return np.clip(np.floor(x), lo, hi).astype(np.int32)


def _empty_prefill(max_blocks):
    return (np.zeros(0, np.int32), np.zeros(0, np.int32),
            np.zeros((0, max_blocks), np.int32))


def make_decode(name, seed, lens, Hq, Hkv, D, P, kv_dtype="bf16",
                max_blocks=None, shared_tokens=0, num_sharers=0,
                num_blocks=None) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 7777))
    lens = np.asarray(lens, dtype=np.int32)
    if max_blocks is None:
        max_blocks = int(_pages(np.array([max(1, int(lens.max()))]), P)[0])
    tables, nb = _allocate(rng, lens, P, max_blocks, shared_tokens,
                           num_sharers, num_blocks)
    pl, pc, pt = _empty_prefill(max_blocks)
    sc = FP8_SCALE if kv_dtype == "fp8_e4m3" else 1.0
    return Workload(name, seed, Hq, Hkv, D, P, kv_dtype, nb, lens, tables,
                    pl, pc, pt, sc, sc, shared_tokens, num_sharers)


def with_head_scales(w: Workload) -> Workload:
    """The same FP8 workload with a different scale per kv head: head h uses
    FP8_SCALE * (1 + 0.37 h) for K and FP8_SCALE * (1 + 0.23 h) for V, so no
    code saturates and heads differ by up to several binades of code range."""
    if w.kv_dtype != "fp8_e4m3":
        raise ValueError("per-head scales apply to FP8 pools")
    h = np.arange(w.num_kv_heads, dtype=np.float64)
    ks = (FP8_SCALE * (1.0 + 0.37 * h)).astype(np.float32)
    vs = (FP8_SCALE * (1.0 + 0.23 * h)).astype(np.float32)
    return dataclasses.replace(w, name=w.name + "_head_scales", k_scales=ks, v_scales=vs)


def make_mixed(name, seed, decode_lens, prior_lens, chunk_lens, Hq, Hkv, D, P,
               max_blocks=None, num_blocks=None, kv_dtype="bf16") -> Workload:
    """Decode sequences plus prefill chunks appended onto prior contexts."""
    rng = np.random.Generator(np.random.PCG64(seed + 7777))
    decode_lens = np.asarray(decode_lens, np.int32)
    prior_lens = np.asarray(prior_lens, np.int32)
    chunk_lens = np.asarray(chunk_lens, np.int32)
    pre_lens = (prior_lens + chunk_lens).astype(np.int32)
    all_lens = np.concatenate([decode_lens, pre_lens])
    if max_blocks is None:
        max_blocks = int(_pages(np.array([int(all_lens.max())]), P)[0])
    tables, nb = _allocate(rng, all_lens, P, max_blocks, num_blocks=num_blocks)
    B = len(decode_lens)
    sc = FP8_SCALE if kv_dtype == "fp8_e4m3" else 1.0
    return Workload(name, seed, Hq, Hkv, D, P, kv_dtype, nb, decode_lens,
                    tables[:B].copy(), pre_lens, chunk_lens, tables[B:].copy(), sc, sc)


def with_fp8_kv(w: Workload) -> Workload:
    """The same batch (lengths, pages, values) with the KV pool stored as FP8
    E4M3 codes under the per-tensor scale FP8_SCALE."""
    return dataclasses.replace(w, name=w.name + "_fp8kv", kv_dtype="fp8_e4m3",
                               k_scale=FP8_SCALE, v_scale=FP8_SCALE)


# -- the five configurations -------------------------------------------------
CONFIG_NAMES = {
    1: "tiny_decode_b4_h8_d64_p16",
    2: "llama2_13b_mha_decode_b64_h40_d128_p64",
    3: "llama3_8b_gqa_decode_b256_h32kv8_d128_p32",
    4: "llama3_70b_gqa_fp8_prefix_decode_b128_h64kv8_d128_p64",
    5: "mixed_prefill4x512_decode32_h32kv8_d128_p32",
    # not one of the five: a longer-context chunked prefill of the same
    # Llama-3-8B GQA shape (8 chunks of 1024 tokens onto prior contexts of
    # 4096), for the prefill kernel's rate away from the mixed step's short
    # contexts
    "long_prefill": "long_prefill_8x1024_prior4096_h32kv8_d128_p32",
    # configuration 5's batch with its KV cache stored as FP8 E4M3
    "mixed_fp8": "mixed_prefill4x512_decode32_h32kv8_d128_p32_fp8kv",
}


def config(i, num_seqs: Optional[int] = None) -> Workload:
    """Configuration i (1..5, or "long_prefill") at full size; seed 31000 + i
    (31006 for the long prefill).

    ``num_seqs`` keeps only the first sequences of the batch (same lengths,
    same shapes, a pool sized for them): a smaller case of the same kernel,
    e.g. for profiler captures."""
    w = _config_full(i)
    if num_seqs is None or num_seqs >= w.num_seqs:
        return w
    lens = w.context_lens[:num_seqs]
    sharers = min(w.num_sharers, num_seqs)
    if w.num_prefill:
        return make_mixed(w.name + f"_first{num_seqs}", w.seed, lens, w.prefill_context_lens
                          - w.prefill_chunk_lens, w.prefill_chunk_lens, w.num_q_heads,
                          w.num_kv_heads, w.head_dim, w.block_size,
                          max_blocks=w.max_blocks_per_seq)
    return make_decode(w.name + f"_first{num_seqs}", w.seed, lens, w.num_q_heads,
                       w.num_kv_heads, w.head_dim, w.block_size, kv_dtype=w.kv_dtype,
                       max_blocks=w.max_blocks_per_seq,
                       shared_tokens=w.shared_prefix_tokens if sharers > 1 else 0,
                       num_sharers=sharers if sharers > 1 else 0)


def _config_full(i) -> Workload:
    if i == "mixed_fp8":
        return with_fp8_kv(_config_full(5))
    if i == "long_prefill":
        n = 8
        return make_mixed(CONFIG_NAMES[i], 31006, np.zeros(0, np.int32),
                          np.full(n, 4096, np.int32), np.full(n, 1024, np.int32), 32, 8, 128, 32,
                          max_blocks=160)
    seed = 31000 + i
    rng = np.random.Generator(np.random.PCG64(seed))
    if i == 1:
        lens = _uniform_int(rng, 1, 64, 4)
        return make_decode(CONFIG_NAMES[1], seed, lens, 8, 8, 64, 16,
                           max_blocks=4, num_blocks=64)
    if i == 2:
        lens = _uniform_int(rng, 128, 4096, 64)
        return make_decode(CONFIG_NAMES[2], seed, lens, 40, 40, 128, 64,
                           max_blocks=64)
    if i == 3:
        lens = _log_uniform_int(rng, 16, 8192, 256)
        return make_decode(CONFIG_NAMES[3], seed, lens, 32, 8, 128, 32,
                           max_blocks=256)
    if i == 4:
        B, sharers, prefix = 128, 64, 2048
        lens = np.empty(B, np.int32)
        # sharers hold the prefix plus at least one private token, so the
        # appended token never lands in a shared page
        lens[:sharers] = _uniform_int(rng, prefix + 1, 32768, sharers)
        lens[sharers:] = _uniform_int(rng, 1024, 32768, B - sharers)
        return make_decode(CONFIG_NAMES[4], seed, lens, 64, 8, 128, 64,
                           kv_dtype="fp8_e4m3", max_blocks=512,
                           shared_tokens=prefix, num_sharers=sharers)
    if i == 5:
        dec = _uniform_int(rng, 256, 4096, 32)
        prior = _uniform_int(rng, 0, 3072, 4)
        chunk = np.full(4, 512, np.int32)
        return make_mixed(CONFIG_NAMES[5], seed, dec, prior, chunk, 32, 8, 128, 32,
                          max_blocks=128)
    raise ValueError(f"unknown config {i}")


def small_config(i: int, variant: int = 0) -> Workload:
    """A reduced batch with the shapes of configuration i (for parity tests).

    Same heads, head_dim, block size and KV dtype; fewer sequences and
    shorter contexts, so the oracle checks every output in seconds while
    still spanning several tiles, split partitions and a ragged last page.
    """
    seed = 32000 + 10 * i + variant
    rng = np.random.Generator(np.random.PCG64(seed))
    if i == 1:
        return config(1)
    if i == 2:
        lens = _uniform_int(rng, 128, 700, 3)
        return make_decode(f"small_{CONFIG_NAMES[2]}", seed, lens, 40, 40, 128, 64)
    if i == 3:
        lens = _log_uniform_int(rng, 16, 3000, 12)
        lens[0] = 2500   # long enough to split at a 1024-token partition
        lens[1] = 1
        return make_decode(f"small_{CONFIG_NAMES[3]}", seed, lens, 32, 8, 128, 32)
    if i == 4:
        B, sharers, prefix = 6, 3, 2048
        lens = np.empty(B, np.int32)
        lens[:sharers] = _uniform_int(rng, prefix + 1, 4000, sharers)
        lens[sharers:] = _uniform_int(rng, 1024, 4000, B - sharers)
        return make_decode(f"small_{CONFIG_NAMES[4]}", seed, lens, 64, 8, 128, 64,
                           kv_dtype="fp8_e4m3", shared_tokens=prefix,
                           num_sharers=sharers)
    if i == 5:
        dec = _uniform_int(rng, 256, 900, 4)
        prior = np.array([0, 333], np.int32)
        chunk = np.array([200, 131], np.int32)
        return make_mixed(f"small_{CONFIG_NAMES[5]}", seed, dec, prior, chunk,
                          32, 8, 128, 32)
    raise ValueError(f"unknown config {i}")
