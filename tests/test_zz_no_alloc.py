"""pkv_paged_attention_noalloc: decode attention for callers that cannot
allocate device memory (a plugin that is handed only its input and output
buffers, or a step that must not call cudaMalloc).  Called here through the
C ABI with raw device pointers.  Its output must match the fp64 oracle
within the decode tolerances, and pkv_paged_attention (which uses a caller
workspace) within the same tolerances, on consecutive calls that reuse the
library's one scratch array with different sizes -- both with a host
synchronisation between calls and with the calls only stream-ordered.

This file sorts last so a run that stops at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import assert_close, device_pools, device_step_inputs, oracle_decode_rows

pytestmark = pytest.mark.gpu


def _noalloc_c(w, d, kp, vp, out, partition, stream=None):
    """Direct C-ABI call: raw pointers, torch's current stream by default."""
    desc = pkv.pool_desc(kp, w.k_scale, w.v_scale)
    s = stream if stream is not None else torch.cuda.current_stream()
    return pkv.lib().pkv_paged_attention_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.byref(desc),
        ctypes.c_void_p(d["block_tables"].data_ptr()), int(d["block_tables"].shape[1]),
        ctypes.c_void_p(d["context_lens"].data_ptr()), w.num_seqs, w.num_q_heads,
        w.max_context_len, float(w.scale), int(partition), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(s.cuda_stream))


def _case(cfg):
    w = W.small_config(cfg)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    return w, d, kp, vp


def _compare(got, ref, fp8):
    err = (got.float() - ref.float()).abs()
    assert torch.isfinite(got.float()).all()
    if fp8:
        assert err.max().item() <= 6e-2
    else:
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3


def _check_oracle(w, out, seqs):
    """Rows of the listed sequences, every kv head, against the fp64 oracle."""
    G = w.group
    fp8 = w.kv_dtype == "fp8_e4m3"
    kn, vn = w.kv_new()
    for h in range(w.num_kv_heads):
        kvh = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
        for s in seqs:
            want = oracle_decode_rows(w, s, h, kvh)
            assert_close(out[s, h * G:(h + 1) * G], want, fp8, f"noalloc {w.name} s={s} h={h}")


def _ref(w, d, kp, vp, part):
    return pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                               w.max_context_len, w.scale, k_scale=w.k_scale,
                               v_scale=w.v_scale, partition_tokens=part)


def test_noalloc_matches_oracle_and_workspace_entry_point_on_consecutive_calls():
    cases = [(_case(3), 64), (_case(4), 0), (_case(3), 128)]
    for (w, d, kp, vp), part in cases:
        ref = _ref(w, d, kp, vp, part)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_c(w, d, kp, vp, out, part) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        _compare(out, ref, w.kv_dtype == "fp8_e4m3")
        _check_oracle(w, out, seqs=[0, w.num_seqs // 2, w.num_seqs - 1])


def test_noalloc_stream_ordered_calls_without_host_sync():
    # three calls of different sizes enqueued back to back on one stream, no
    # synchronisation between them: stream order alone keeps each call's use
    # of the shared scratch apart from the next one's
    cases = [(_case(3), 64), (_case(2), 0), (_case(4), 128)]
    refs = [_ref(w, d, kp, vp, part) for (w, d, kp, vp), part in cases]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    outs = [torch.full_like(r, float("nan")) for r in refs]
    torch.cuda.synchronize()
    for ((w, d, kp, vp), part), out in zip(cases, outs):
        assert _noalloc_c(w, d, kp, vp, out, part, stream=side) == pkv.PKV_OK
    side.synchronize()
    assert pkv.get_device_error() == 0
    for ((w, d, kp, vp), part), out, ref in zip(cases, outs, refs):
        _compare(out, ref, w.kv_dtype == "fp8_e4m3")
        _check_oracle(w, out, seqs=[0, w.num_seqs - 1])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w, d, kp, vp = _case(3)
    limit = pkv.lib().pkv_paged_attention_noalloc_max_scratch()
    assert pkv.paged_attention_workspace_size(4096, 64, 32768, kp, 64) > limit
    out = torch.zeros_like(d["q"])
    desc = pkv.pool_desc(kp)
    st = pkv.lib().pkv_paged_attention_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.byref(desc),
        ctypes.c_void_p(d["block_tables"].data_ptr()), 512,
        ctypes.c_void_p(d["context_lens"].data_ptr()), 4096, 64, 32768, 0.1, 64,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3  # PKV_ERR_WORKSPACE: nothing enqueued
    torch.cuda.synchronize()
    assert out.float().abs().sum().item() == 0
