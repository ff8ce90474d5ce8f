"""Paged decode attention on the GPU against the fp64 oracle.

Small batches of every configuration's shape are checked element by element;
full-size configurations are checked on sampled (sequence, kv head) rows in
the launch configuration the benchmark times (automatic split plan).
Tolerances: bf16 KV max |err| <= 2e-2 and mean |err| <= 2e-3; FP8 KV max
|err| <= 6e-2 (against the oracle run on the same stored FP8 codes).
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import (assert_close, device_pools, device_step_inputs,
                              oracle_decode_rows)

pytestmark = pytest.mark.gpu


def _run_step(w, d, k_pool, v_pool, partition=0):
    ks, vs = w.scale_tensors(d["q"].device)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], k_pool, v_pool, w.k_scale, w.v_scale,
                  k_scales=ks, v_scales=vs)
    return pkv.paged_attention(d["q"], k_pool, v_pool, d["block_tables"], d["context_lens"],
                               w.max_context_len, w.scale, k_scale=w.k_scale,
                               v_scale=w.v_scale, partition_tokens=partition,
                               k_scales=ks, v_scales=vs)


def _check_all_rows(w, out, seqs=None, heads=None):
    G = w.group
    fp8 = w.kv_dtype == "fp8_e4m3"
    kn, vn = w.kv_new()
    cache = {}
    seqs = range(w.num_seqs) if seqs is None else seqs
    worst = 0.0
    for s in seqs:
        for h in (range(w.num_kv_heads) if heads is None else heads):
            if h not in cache:
                cache[h] = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
            want = oracle_decode_rows(w, s, h, cache[h])
            mx, _ = assert_close(out[s, h * G:(h + 1) * G], want, fp8, f"{w.name} s={s} h={h}")
            worst = max(worst, mx)
    return worst


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_small_configs_every_row(cfg):
    w = W.small_config(cfg)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out)


@pytest.mark.parametrize("partition", [0, 64, 128, 1024, 2048])
def test_split_partitions_agree_with_oracle(partition):
    w = W.small_config(3)                     # lens up to 2500: 1..40 partitions
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp, partition)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out, heads=[0, 5])


@pytest.mark.parametrize("G,D,P", [(1, 64, 16), (2, 128, 32), (4, 64, 64), (8, 128, 16),
                                   (8, 64, 32), (1, 128, 64), (4, 128, 64), (8, 128, 32),
                                   (1, 128, 128), (8, 128, 128), (2, 64, 128)])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_shapes_and_ragged_lengths(G, D, P, kv_dtype):
    # lengths around tile (16), page and partition boundaries, plus 0 and 1
    lens = [0, 1, 15, 16, 17, P - 1, P, P + 1, 3 * P + 5, 511, 512, 513, 1500]
    hkv = 2
    w = W.make_decode(f"edge_G{G}_D{D}_P{P}_{kv_dtype}", 555 + G + D + P,
                      np.maximum(lens, 1), hkv * G, hkv, D, P, kv_dtype=kv_dtype)
    w.context_lens = np.array(lens, np.int32)  # a zero-length row: no token appended
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp, partition=512)
    assert pkv.get_device_error() == 0
    assert torch.all(out[0].float() == 0)
    _check_all_rows(w, out, seqs=range(1, len(lens)))


@pytest.mark.parametrize("G,D,P", [(8, 128, 32), (4, 128, 16), (2, 128, 32), (8, 64, 16)])
@pytest.mark.parametrize("partition", [0, 256])
def test_fp8_per_head_scales(G, D, P, partition):
    # per-kv-head K and V scales through both decode paths (tensor-core for
    # D=128 with 4-8 packed heads, CUDA cores otherwise) and through the merge
    lens = [1, 17, P + 3, 300, 777, 1500]
    hkv = 4
    w = W.with_head_scales(W.make_decode(f"heads_G{G}_D{D}_P{P}", 880 + G + D + P, lens,
                                         hkv * G, hkv, D, P, kv_dtype="fp8_e4m3"))
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp, partition=partition)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out)


def test_fp8_per_head_scales_prefix_sharing_config():
    w = W.with_head_scales(W.small_config(4))
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out, heads=[0, 3, 7])


def test_full_block_table_capacity():
    # sequences that fill every entry of their block-table row
    P, maxb = 32, 24
    w = W.make_decode("full_table", 777, [P * maxb, P * maxb - 3], 8, 2, 128, P, max_blocks=maxb)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp, partition=256)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out)


@pytest.mark.parametrize("cfg", [2, 4])
def test_bad_page_id_is_reported_not_dereferenced(cfg):
    w = W.small_config(cfg)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    bt = d["block_tables"].clone()
    bt[1, 2] = w.num_blocks + 1000             # far outside the pool
    bt[2, 0] = -7
    pkv.paged_attention(d["q"], kp, vp, bt, d["context_lens"], w.max_context_len, w.scale,
                        k_scale=w.k_scale, v_scale=w.v_scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    # a clean call afterwards is unaffected
    out = _run_step(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check_all_rows(w, out, seqs=[0, 1], heads=[3])


def test_context_len_beyond_declared_max_is_reported():
    w = W.small_config(2)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                        int(w.context_lens.max()) - 5, w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS


def test_repeatable_bitwise():
    w = W.small_config(3)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    a = _run_step(w, d, kp, vp).clone()
    b = _run_step(w, d, kp, vp).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _sample_rows(w, n_seqs=6, seed=0):
    rng = np.random.default_rng(seed)
    L = w.context_lens
    picks = {int(np.argmax(L)), int(np.argmin(L))}
    if w.num_sharers:
        picks |= {0, w.num_sharers}
    while len(picks) < n_seqs:
        picks.add(int(rng.integers(0, w.num_seqs)))
    return sorted(picks), [int(rng.integers(0, w.num_kv_heads)) for _ in picks]


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_sampled_rows(cfg):
    w = W.config(cfg)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _run_step(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    seqs, heads = _sample_rows(w)
    for s, h in zip(seqs, heads):
        _check_all_rows(w, out, seqs=[s], heads=[h])
    del kp, vp
    torch.cuda.empty_cache()
