"""Input generator: determinism, structure of block tables and slot maps."""
import numpy as np
import pytest
import torch

import workloads as W


def test_values_deterministic_and_unit_normal():
    a = W.dense_values(5, "k", (1 << 20,))
    b = W.dense_values(5, "k", (1 << 20,))
    c = W.dense_values(6, "k", (1 << 20,))
    d = W.dense_values(5, "v", (1 << 20,))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a, c) and not torch.equal(a, d)
    f = a.float()
    assert abs(f.mean().item()) < 5e-3 and abs(f.std().item() - 1) < 5e-3
    assert f.abs().max().item() <= W.VALUE_BOUND


def test_pool_values_index_is_row_major_pool_index():
    hkv, P, D = 3, 4, 8
    whole = W.dense_values(9, "k", (10, hkv, P, D))
    some = W.pool_values(9, "k", [7, 2], hkv, P, D)
    assert torch.equal(some[0].view(torch.int16), whole[7].view(torch.int16))
    assert torch.equal(some[1].view(torch.int16), whole[2].view(torch.int16))
    # high index bits matter (pools beyond 2^32 elements)
    big = torch.tensor([5, 5 + (1 << 32)], dtype=torch.int64)
    v = W.normal_bf16(1, "k", big)
    assert v[0].item() != v[1].item()


@pytest.mark.parametrize("i", [1, 2, 3, 4, 5])
def test_config_structure(i):
    w = W.config(i)
    w2 = W.config(i)
    assert np.array_equal(w.context_lens, w2.context_lens)
    assert np.array_equal(w.block_tables, w2.block_tables)
    P = w.block_size
    tables = [(w.block_tables, w.context_lens)]
    if w.num_prefill:
        tables.append((w.prefill_block_tables, w.prefill_context_lens))
    used = []
    for bt, cl in tables:
        for s in range(len(cl)):
            n = (int(cl[s]) + P - 1) // P
            row = bt[s]
            assert np.all(row[:n] >= 0) and np.all(row[:n] < w.num_blocks)
            assert np.all(row[n:] == -1)
            used.append(row[:n])
    allp = np.concatenate(used)
    shared = w.shared_prefix_tokens // P if w.num_sharers else 0
    # pages are private except the shared prefix, which sharers reuse
    uniq = len(np.unique(allp))
    assert uniq == len(allp) - shared * max(0, w.num_sharers - 1)
    assert w.num_blocks >= uniq
    if i != 1:
        assert w.num_blocks == int(np.ceil(1.25 * uniq))
    # the appended tokens land in distinct slots of the right pages
    slots = w.append_slot_mapping()
    assert len(np.unique(slots)) == len(slots)
    assert np.all(slots >= 0) and np.all(slots < w.num_blocks * P)


def test_config_distributions():
    w2 = W.config(2)
    assert w2.context_lens.min() >= 128 and w2.context_lens.max() <= 4096
    w3 = W.config(3)
    assert w3.context_lens.min() >= 16 and w3.context_lens.max() <= 8192
    assert 0.1 < np.mean(w3.context_lens > 2048) < 0.35   # log-uniform mix
    w4 = W.config(4)
    assert w4.kv_dtype == "fp8_e4m3" and w4.num_sharers == 64
    assert np.all(w4.block_tables[:64, :32] == w4.block_tables[0, :32])
    assert np.all(w4.context_lens[:64] > 2048)
    w5 = W.config(5)
    assert w5.num_prefill == 4 and np.all(w5.prefill_chunk_lens == 512)
    assert np.all(w5.prefill_context_lens >= 512)
    assert np.all(w5.prefill_context_lens <= 3072 + 512)


def test_decode_slot_is_last_position():
    w = W.small_config(3)
    slots = w.decode_slot_mapping()
    P = w.block_size
    for s, L in enumerate(w.context_lens):
        assert slots[s] // P == w.block_tables[s, (L - 1) // P]
        assert slots[s] % P == (L - 1) % P


def test_prefill_slots_cover_chunk_positions():
    w = W.small_config(5)
    slots = w.prefill_slot_mapping()
    cu = w.cu_seqlens_q()
    P = w.block_size
    for s in range(w.num_prefill):
        L, C = int(w.prefill_context_lens[s]), int(w.prefill_chunk_lens[s])
        for i, pos in enumerate(range(L - C, L)):
            sl = slots[cu[s] + i]
            assert sl // P == w.prefill_block_tables[s, pos // P] and sl % P == pos % P


@pytest.mark.gpu
def test_generator_identical_on_gpu():
    idx = torch.arange(0, 1 << 22, dtype=torch.int64) * 977 + (3 << 32)
    cpu = W.normal_bf16(31002, "k", idx)
    gpu = W.normal_bf16(31002, "k", idx.cuda()).cpu()
    assert torch.equal(cpu.view(torch.int16), gpu.view(torch.int16))


def test_head_scales_workload():
    w = W.with_head_scales(W.small_config(4))
    assert w.k_scales.dtype == np.float32 and w.k_scales.shape == (w.num_kv_heads,)
    assert w.head_scales(0) == (float(np.float32(W.FP8_SCALE)), float(np.float32(W.FP8_SCALE)))
    assert w.head_scales(3)[0] > w.head_scales(3)[1] > w.head_scales(0)[1]
    ks, vs = w.scale_tensors()
    assert ks.dtype == torch.float32 and torch.equal(ks, torch.from_numpy(w.k_scales))
    assert W.small_config(4).scale_tensors() == (None, None)
    with pytest.raises(ValueError):
        W.with_head_scales(W.small_config(3))
