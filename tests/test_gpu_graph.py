"""The decode step (kv_append + paged attention) captured in a CUDA graph and
replayed gives bit-identical results to eager launches: every call is
stream-ordered and synchronises nothing, so a batch-size bucket can be
captured once and replayed each step ("TensorRT-LLM框架解析与高性能推理优化实践"
§8.1, "CUDA Graph优化")."""
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import device_pools, device_step_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 3])
def test_graph_replay_matches_eager(cfg):
    w = W.small_config(cfg)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    B, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    ws = torch.empty(pkv.paged_attention_workspace_size(B, Hq, w.max_context_len, kp, 64),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")

    def step():
        pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
        pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                            w.max_context_len, w.scale, out=out, workspace=ws,
                            partition_tokens=64)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # first call: per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("fp8", [False, True])
def test_mixed_step_graph_replay_matches_eager(fp8):
    # one mixed iteration: the append of every new row, the chunked prefill
    # and the decode call, captured once; over an FP8 pool with per-head
    # scales too (the prefill converts its codes inside the kernel)
    w = W.small_config(5)
    if fp8:
        w = W.with_head_scales(W.with_fp8_kv(w))
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    ks, vs = w.scale_tensors("cuda")
    B, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    ws = torch.empty(pkv.paged_attention_workspace_size(B, Hq, w.max_context_len, kp, 128),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    out_p = torch.empty_like(d["q_prefill"])
    sc = dict(k_scale=w.k_scale, v_scale=w.v_scale, k_scales=ks, v_scales=vs)

    def step():
        pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, **sc)
        pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp, d["prefill_block_tables"],
                          d["prefill_context_lens"], int(w.prefill_chunk_lens.max()), w.scale,
                          out=out_p, **sc)
        pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                            w.max_context_len, w.scale, out=out, workspace=ws,
                            partition_tokens=128, **sc)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                  # first calls: per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager, eager_p = out.clone(), out_p.clone()
    out.zero_()
    out_p.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert torch.equal(out_p.view(torch.int16), eager_p.view(torch.int16))
