"""pkv_paged_attention_append (the step's appends fused into the attention's
planning launch) against the two-call path and the oracle.

The fused call runs the same kernels on the same data as pkv_kv_append
followed by pkv_paged_attention, so pools and outputs must agree bit for bit
with the two-call path; rows are also checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import assert_close, device_pools, device_step_inputs, oracle_decode_rows

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _both_paths(w, partition=0):
    d = device_step_inputs(w)
    ks, vs = w.scale_tensors("cuda")
    kp1, vp1 = device_pools(w)
    kp2, vp2 = kp1.clone(), vp1.clone()
    kw = dict(k_scale=w.k_scale, v_scale=w.v_scale, k_scales=ks, v_scales=vs)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp1, vp1, **kw)
    ref = pkv.paged_attention(d["q"], kp1, vp1, d["block_tables"], d["context_lens"],
                              w.max_context_len, w.scale, partition_tokens=partition, **kw)
    out = pkv.paged_attention_append(d["q"], d["k_new"], d["v_new"], d["slots"], kp2, vp2,
                                     d["block_tables"], d["context_lens"], w.max_context_len,
                                     w.scale, partition_tokens=partition, **kw)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return d, (kp1, vp1, ref), (kp2, vp2, out)


@pytest.mark.parametrize("cfg,head_scales", [(1, False), (2, False), (3, False), (4, False),
                                             (4, True)])
def test_fused_equals_two_calls_and_oracle(cfg, head_scales):
    w = W.small_config(cfg)
    if head_scales:
        w = W.with_head_scales(w)
    d, (kp1, vp1, ref), (kp2, vp2, out) = _both_paths(w)
    assert torch.equal(_bits(kp1), _bits(kp2)) and torch.equal(_bits(vp1), _bits(vp2))
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    G = w.group
    for s in (0, w.num_seqs - 1):
        for h in (0, w.num_kv_heads - 1):
            want = oracle_decode_rows(w, s, h)
            assert_close(out[s, h * G:(h + 1) * G], want, w.kv_dtype == "fp8_e4m3",
                         f"{w.name} s={s} h={h}")


@pytest.mark.parametrize("partition", [64, 256])
def test_fused_with_split_partitions(partition):
    w = W.small_config(3)
    _, (kp1, vp1, ref), (kp2, vp2, out) = _both_paths(w, partition)
    assert torch.equal(kp1.view(torch.int16), kp2.view(torch.int16))
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))


def test_fused_degenerate_counts():
    w = W.small_config(2)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    # no new tokens: a plain attention call
    none = torch.zeros(0, dtype=torch.int64, device="cuda")
    empty = torch.zeros((0, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    a = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                            w.max_context_len, w.scale)
    b = pkv.paged_attention_append(d["q"], empty, empty, none, kp, vp, d["block_tables"],
                                   d["context_lens"], w.max_context_len, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # no sequences: a plain append
    kp2, vp2 = device_pools(w)
    kp3, vp3 = kp2.clone(), vp2.clone()
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp2, vp2)
    q0 = torch.zeros((0, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_append(q0, d["k_new"], d["v_new"], d["slots"], kp3, vp3,
                               d["block_tables"][:0], d["context_lens"][:0], 0, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(kp2.view(torch.int16), kp3.view(torch.int16))


def test_fused_out_of_pool_slot_is_reported_and_skipped():
    w = W.small_config(3)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    before = kp.clone()
    slots = d["slots"].clone()
    slots[0] = w.num_blocks * w.block_size + 5          # past the pool
    pkv.paged_attention_append(d["q"], d["k_new"], d["v_new"], slots, kp, vp,
                               d["block_tables"], d["context_lens"], w.max_context_len, w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    # every other token was appended
    page, off = int(d["slots"][1]) // w.block_size, int(d["slots"][1]) % w.block_size
    assert torch.equal(kp[page, :, off].view(torch.int16),
                       d["k_new"][1].view(torch.int16))
    page0, off0 = int(d["slots"][0]) // w.block_size, int(d["slots"][0]) % w.block_size
    assert torch.equal(kp[page0, :, off0].view(torch.int16), before[page0, :, off0].view(torch.int16))


def test_fused_step_in_a_cuda_graph():
    w = W.small_config(3)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = torch.empty_like(d["q"])
    ws = torch.empty(pkv.paged_attention_workspace_size(w.num_seqs, w.num_q_heads,
                                                        w.max_context_len, kp), dtype=torch.uint8,
                     device="cuda")
    step = lambda: pkv.paged_attention_append(d["q"], d["k_new"], d["v_new"], d["slots"], kp, vp,
                                              d["block_tables"], d["context_lens"],
                                              w.max_context_len, w.scale, out=out, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
