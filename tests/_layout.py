"""Test-side helpers: lay dense per-sequence K/V into a paged pool.

This is the test's own construction (the inverse of a gather), written
independently of the oracle, so a wrong index in the oracle's gather shows up
as a mismatch against dense attention.
"""
import numpy as np
import torch


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (via torch, RNE) and return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paginate(dense_seqs, P, num_blocks, rng, pool_dtype=np.uint16, fill=0):
    """dense_seqs: list of [L_s, Hkv, D] arrays.  Returns pool, block_tables.

    Each sequence gets ceil(L/P) distinct random pages; token i of a sequence
    is written to page table[i // P] at offset i % P.
    """
    Hkv, D = dense_seqs[0].shape[1:]
    need = [(x.shape[0] + P - 1) // P for x in dense_seqs]
    maxb = max(1, max(need))
    ids = rng.permutation(num_blocks)
    assert sum(need) <= num_blocks
    pool = np.full((num_blocks, Hkv, P, D), fill, dtype=pool_dtype)
    tables = np.full((len(dense_seqs), maxb), -1, np.int32)
    cur = 0
    for s, x in enumerate(dense_seqs):
        for j in range(need[s]):
            page = ids[cur]
            cur += 1
            tables[s, j] = page
            chunk = x[j * P:(j + 1) * P]            # [<=P, Hkv, D]
            pool[page, :, :chunk.shape[0], :] = chunk.transpose(1, 0, 2)
    return pool, tables


def dense_attention(q, K, V, scale, mask=None):
    """torch SDPA in fp64.  q [Hq, M, D], K/V [Hkv, L, D] -> [Hq, M, D].

    GQA by torch's repeat_interleave convention (q head a -> kv head a//G).
    """
    q = torch.as_tensor(q, dtype=torch.float64)
    K = torch.as_tensor(K, dtype=torch.float64)
    V = torch.as_tensor(V, dtype=torch.float64)
    G = q.shape[0] // K.shape[0]
    K = K.repeat_interleave(G, dim=0)
    V = V.repeat_interleave(G, dim=0)
    m = None if mask is None else torch.as_tensor(mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None], K[None], V[None], attn_mask=m, scale=scale)
    return out[0].numpy()
