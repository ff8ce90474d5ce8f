"""Decode attention at the edges of its inputs, against the fp64 oracle.

* q far from N(0, 1): bf16 q scaled by 300 and by 1e-5 (plain softmax
  scale), and by 2^16 and 2^-20 with the softmax scale divided by the same
  power of two, so the scores stay O(1) while q itself sits far outside
  f16's range (|q| up to 3.2e5) or deep in its subnormals.  Every
  decode kernel takes these inputs: the CUDA-core kernel (1-2 packed heads)
  and the tensor-core kernel (4-8 packed heads at head_dim 128), bf16 and FP8
  KV ("TensorRT-LLM框架解析与高性能推理优化实践" §6.2 Paged Attention优化, §7.2
  KV Cache量化: the quantised cache is dequantised inside the kernel, q stays
  in its own precision).
* never-written slots: every slot past a sequence's last token in its last
  page holds a NaN bit pattern (bf16 NaN; E4M3 0x7F / 0xFF); the output must
  not see them, with and without split partitions.
Tolerances as everywhere: bf16 KV max |err| <= 2e-2, mean <= 2e-3; FP8 KV max
|err| <= 6e-2.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import assert_close, device_pools, device_step_inputs, oracle_decode_rows

pytestmark = pytest.mark.gpu

# (packed heads G, head_dim, block size): CUDA-core kernel for G 1-2 or
# head_dim 64, tensor-core kernel for G 4-8 at head_dim 128
KERNEL_SHAPES = [(1, 128, 64), (2, 64, 32), (4, 128, 32), (8, 128, 16), (8, 64, 64)]
LENS = [1, 7, 16, 33, 130, 511, 777, 1300]


def _workload(tag, G, D, P, kv_dtype, seed):
    hkv = 2
    return W.make_decode(f"{tag}_G{G}_D{D}_P{P}_{kv_dtype}", seed, LENS, hkv * G, hkv, D, P,
                         kv_dtype=kv_dtype)


def _check(w, out, q_host=None, scale=None):
    G = w.group
    fp8 = w.kv_dtype == "fp8_e4m3"
    kn, vn = w.kv_new()
    for h in range(w.num_kv_heads):
        kvh = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
        for s in range(w.num_seqs):
            want = oracle_decode_rows(w, s, h, kvh, q_host=q_host, scale=scale)
            assert_close(out[s, h * G:(h + 1) * G], want, fp8, f"{w.name} s={s} h={h}")


@pytest.mark.parametrize("mult,scale_div", [(300.0, 1.0), (1e-5, 1.0), (2.0 ** 16, 2.0 ** 16),
                                            (2.0 ** -20, 2.0 ** -20)])
@pytest.mark.parametrize("G,D,P", KERNEL_SHAPES)
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_q_far_from_unit_scale(mult, scale_div, G, D, P, kv_dtype):
    w = _workload("qrange", G, D, P, kv_dtype, 4100 + G + D + P)
    # the scaled q is formed on the host (fp32 product, then RNE to bf16) and
    # the same bf16 values feed the oracle and the kernels
    q_host = (w.q_decode().float() * mult).to(torch.bfloat16)
    scale = w.scale / scale_div
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    q = q_host.to("cuda")
    for partition in (0, 256):
        pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
        out = pkv.paged_attention(q, kp, vp, d["block_tables"], d["context_lens"],
                                  w.max_context_len, scale, k_scale=w.k_scale,
                                  v_scale=w.v_scale, partition_tokens=partition)
        assert pkv.get_device_error() == 0
        _check(w, out, q_host=q_host, scale=scale)


def _poison_tails(w, kp, vp):
    """NaN bit patterns in every slot past each sequence's last token, in its
    last page (after this step's append wrote the token at L - 1)."""
    P = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        off = L % P
        if L == 0 or off == 0:
            continue
        last = int(w.block_tables[s, (L - 1) // P])
        if w.kv_dtype == "bf16":
            kp[last, :, off:, :] = float("nan")
            vp[last, :, off:, :] = float("nan")
        else:  # E4M3 NaN codes, both signs
            for pool in (kp, vp):
                pool[last, :, off:, 0::2] = 0x7F
                pool[last, :, off:, 1::2] = 0xFF


@pytest.mark.parametrize("G,D,P", KERNEL_SHAPES)
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("partition", [0, 128])
def test_never_written_slots_past_the_end_do_not_leak(G, D, P, kv_dtype, partition):
    w = _workload("nantail", G, D, P, kv_dtype, 4300 + G + D + P)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    _poison_tails(w, kp, vp)
    out = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                              w.max_context_len, w.scale, k_scale=w.k_scale, v_scale=w.v_scale,
                              partition_tokens=partition)
    assert pkv.get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    _check(w, out)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_never_written_slots_fused_step(kv_dtype):
    # the same through pkv_paged_attention_append: the tails are poisoned
    # before the step, away from the slot the step's own append writes
    w = _workload("nantail_fused", 8, 128, 32, kv_dtype, 4444)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    _poison_tails(w, kp, vp)
    out = pkv.paged_attention_append(d["q"], d["k_new"], d["v_new"], d["slots"], kp, vp,
                                     d["block_tables"], d["context_lens"], w.max_context_len,
                                     w.scale, k_scale=w.k_scale, v_scale=w.v_scale)
    assert pkv.get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    _check(w, out)


@pytest.mark.parametrize("G,D,P", [(8, 128, 32), (4, 128, 16), (2, 128, 64)])
def test_q_range_with_per_head_fp8_scales(G, D, P):
    # the per-head q scaling of the tensor-core decode combined with per-kv-head
    # K / V scales (both multiply the same scores), q at 2^16 with the softmax
    # scale divided by 2^16
    hkv = 4
    w = W.with_head_scales(W.make_decode(f"qrange_heads_G{G}_D{D}_P{P}", 4700 + G + P, LENS,
                                         hkv * G, hkv, D, P, kv_dtype="fp8_e4m3"))
    q_host = (w.q_decode().float() * 2.0 ** 16).to(torch.bfloat16)
    scale = w.scale / 2.0 ** 16
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    ks, vs = w.scale_tensors("cuda")
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale,
                  k_scales=ks, v_scales=vs)
    out = pkv.paged_attention(q_host.to("cuda"), kp, vp, d["block_tables"], d["context_lens"],
                              w.max_context_len, scale, k_scale=w.k_scale, v_scale=w.v_scale,
                              partition_tokens=256, k_scales=ks, v_scales=vs)
    assert pkv.get_device_error() == 0
    _check(w, out, q_host=q_host, scale=scale)
