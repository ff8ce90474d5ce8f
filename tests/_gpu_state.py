"""GPU-test helpers: the oracle-side state of one (sequence, kv head)
rebuilt on the host from the seeded generator (never from the CUDA path),
the tolerance check, and the device inputs (from device_inputs.py).
"""
import numpy as np
import torch

import oracle
import workloads as W
from device_inputs import device_pools, device_step_inputs  # noqa: F401  (re-exported)

BF16_MAX_ABS, BF16_MEAN_ABS, FP8_MAX_ABS = 2e-2, 2e-3, 6e-2


def host_head_pools(w: W.Workload, page_ids, h: int, k_new_h=None, v_new_h=None):
    """Oracle pools [n, 1, P, D] for kv head h of the given pages, after this
    step's appends: the generator's values, then oracle.kv_append of every
    appended token whose slot falls in these pages."""
    page_ids = np.asarray(page_ids, np.int64)
    P, D = w.block_size, w.head_dim
    ks, vs = w.head_scales(h)
    n = len(page_ids)
    src = {c: W.bf16_bits(W.pool_values_head(w.seed, c, page_ids, h, w.num_kv_heads, P, D))
           for c in ("k", "v")}
    dt = np.uint16 if w.kv_dtype == "bf16" else np.uint8
    kp = np.zeros((n, 1, P, D), dt)
    vp = np.zeros((n, 1, P, D), dt)
    # initial contents: every slot of these pages
    oracle.kv_append(src["k"].reshape(n * P, 1, D), src["v"].reshape(n * P, 1, D),
                     np.arange(n * P, dtype=np.int64), kp, vp, w.kv_dtype, ks, vs)
    # this step's appends that land in these pages
    slots = w.append_slot_mapping()
    if k_new_h is None:
        kn, vn = w.kv_new()
        k_new_h = W.bf16_bits(kn[:, h, :])
        v_new_h = W.bf16_bits(vn[:, h, :])
    where = {int(p): i for i, p in enumerate(page_ids)}
    sel = [t for t in range(len(slots)) if int(slots[t]) // P in where]
    if sel:
        sel = np.array(sel)
        mapped = np.array([where[int(slots[t]) // P] * P + int(slots[t]) % P for t in sel], np.int64)
        oracle.kv_append(k_new_h[sel][:, None, :], v_new_h[sel][:, None, :], mapped, kp, vp,
                         w.kv_dtype, ks, vs)
    return kp, vp


def oracle_decode_rows(w: W.Workload, s: int, h: int, kv_new_h=None, q_host=None,
                       scale=None):
    """fp64 oracle output [G, D] of decode sequence s, q heads of kv head h.

    q_host (bf16 CPU tensor [B, Hq, D]) and scale replace the workload's own
    q and softmax scale when given."""
    L = int(w.context_lens[s])
    P = w.block_size
    npg = (L + P - 1) // P
    pages = w.block_tables[s, :npg]
    kp, vp = host_head_pools(w, pages, h, *(kv_new_h or (None, None)))
    G = w.group
    qa = w.q_decode() if q_host is None else q_host
    q = W.bf16_bits(qa[s, h * G:(h + 1) * G, :])[None]
    table = np.arange(max(npg, 1), dtype=np.int32)[None]
    ks, vs = w.head_scales(h)
    out = oracle.paged_attention(q, kp, vp, table, np.array([L], np.int32),
                                 w.scale if scale is None else scale, w.kv_dtype, ks, vs)
    return out[0]


def oracle_prefill_rows(w: W.Workload, s: int, h: int, kv_new_h=None):
    """fp64 oracle output [C, G, D] of prefill sequence s, q heads of kv head h."""
    L = int(w.prefill_context_lens[s])
    C = int(w.prefill_chunk_lens[s])
    P = w.block_size
    npg = (L + P - 1) // P
    pages = w.prefill_block_tables[s, :npg]
    kp, vp = host_head_pools(w, pages, h, *(kv_new_h or (None, None)))
    G = w.group
    cu = w.cu_seqlens_q()
    q = W.bf16_bits(w.q_prefill()[cu[s]:cu[s + 1], h * G:(h + 1) * G, :])
    table = np.arange(max(npg, 1), dtype=np.int32)[None]
    ks, vs = w.head_scales(h)
    out = oracle.paged_prefill(q, np.array([0, C], np.int32), kp, vp, table,
                               np.array([L], np.int32), w.scale, w.kv_dtype, ks, vs)
    return out


def oracle_prefill_window(w: W.Workload, s: int, h: int, r0: int, r1: int, kv_new_h=None):
    """fp64 oracle output [r1 - r0, G, D] of rows r0 .. r1-1 of prefill
    sequence s's chunk, q heads of kv head h: those rows are the last r1 - r0
    tokens of the same sequence cut at length L - C + r1, so the oracle runs
    on that shorter sequence (its first pages, the window's q rows)."""
    L = int(w.prefill_context_lens[s])
    C = int(w.prefill_chunk_lens[s])
    assert 0 <= r0 < r1 <= C
    Lw = L - C + r1
    P = w.block_size
    npg = (Lw + P - 1) // P
    pages = w.prefill_block_tables[s, :npg]
    kp, vp = host_head_pools(w, pages, h, *(kv_new_h or (None, None)))
    G = w.group
    cu = w.cu_seqlens_q()
    q = W.bf16_bits(w.q_prefill()[cu[s] + r0:cu[s] + r1, h * G:(h + 1) * G, :])
    table = np.arange(max(npg, 1), dtype=np.int32)[None]
    ks, vs = w.head_scales(h)
    return oracle.paged_prefill(q, np.array([0, r1 - r0], np.int32), kp, vp, table,
                                np.array([Lw], np.int32), w.scale, w.kv_dtype, ks, vs)


def assert_close(got_bf16: torch.Tensor, want: np.ndarray, fp8: bool, what=""):
    got = got_bf16.detach().float().cpu().numpy().astype(np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    if fp8:
        assert err.max() <= FP8_MAX_ABS, f"{what}: max abs err {err.max():.3g}"
    else:
        assert err.max() <= BF16_MAX_ABS, f"{what}: max abs err {err.max():.3g}"
        assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean abs err {err.mean():.3g}"
    return float(err.max()), float(err.mean())
