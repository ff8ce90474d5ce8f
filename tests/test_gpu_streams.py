"""Calls enqueued on a stream other than torch's current one.  The binding
allocates a call's default output and workspace on the call's own stream,
so the caching allocator cannot hand that memory to an allocation on the
current stream while the call's kernels still run.  Here the side stream is
held back behind a long fill, the call is enqueued on it, and the current
stream at once allocates and writes tensors of the workspace's size; the
call's output must still match the fp64 oracle.  The failure-path self-test
on a side stream must return the kernel's results, not the buffer's fill."""
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import assert_close, device_pools, device_step_inputs, oracle_decode_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("call", ["paged_attention", "paged_attention_append"])
def test_side_stream_call_survives_reallocation_on_the_current_stream(call):
    w = W.small_config(3)                       # long contexts: split partitions and a merge
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    part = 64
    if call == "paged_attention":
        pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    ws_bytes = pkv.paged_attention_workspace_size(w.num_seqs, w.num_q_heads, w.max_context_len,
                                                  kp, part)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    hold = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(side):
        for i in range(6):                      # a few ms of work ahead of the call
            hold.fill_(i)
    if call == "paged_attention":
        out = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                                  w.max_context_len, w.scale, partition_tokens=part,
                                  stream=side)
    else:
        out = pkv.paged_attention_append(d["q"], d["k_new"], d["v_new"], d["slots"], kp, vp,
                                         d["block_tables"], d["context_lens"],
                                         w.max_context_len, w.scale, partition_tokens=part,
                                         stream=side)
    # the call's workspace is already released on the host side: same-size
    # allocations on the current stream, written at once
    junk = [torch.full((ws_bytes,), 255, dtype=torch.uint8, device="cuda") for _ in range(4)]
    junk += [torch.full_like(d["q"], float("nan")) for _ in range(4)]
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    G = w.group
    for s in (0, w.num_seqs // 2, w.num_seqs - 1):
        for h in (0, w.num_kv_heads - 1):
            assert_close(out[s, h * G:(h + 1) * G], oracle_decode_rows(w, s, h), False,
                         f"{call} s={s} h={h}")
    del junk, hold


def test_self_test_on_a_side_stream_reads_the_kernels_results():
    side = torch.cuda.Stream()
    hold = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(side):
        for i in range(4):
            hold.fill_(i)
    res = pkv.self_test_bounded_wait(2_000_000, stream=side)
    assert res == [0, 0, 1, 1, 1], res
    assert pkv.get_device_error(stream=side) == pkv.PKV_ERR_DEVICE_TIMEOUT
    assert pkv.get_device_error() == 0
