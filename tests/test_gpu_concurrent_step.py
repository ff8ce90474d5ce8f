"""The mixed step's decode call and prefill call on two streams (the decode
on a high-priority stream, both after one append of the step's rows) give
exactly the outputs of the same calls run one after the other, and the
oracle's rows."""
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import (assert_close, device_pools, device_step_inputs,
                              oracle_decode_rows)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg_variant", [0, 1])
def test_two_streams_match_one_stream(cfg_variant):
    w = W.small_config(5, cfg_variant)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    maxq = int(w.prefill_chunk_lens.max())

    def decode(stream=None):
        return pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                                   w.max_context_len, w.scale, stream=stream)

    def prefill(stream=None):
        return pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp,
                                 d["prefill_block_tables"], d["prefill_context_lens"], maxq,
                                 w.scale, stream=stream)

    want_d, want_p = decode(), prefill()
    main = torch.cuda.current_stream()
    hi = torch.cuda.Stream(priority=-1)
    for _ in range(3):
        start, done = torch.cuda.Event(), torch.cuda.Event()
        start.record(main)
        hi.wait_event(start)
        got_p = prefill()
        with torch.cuda.stream(hi):
            got_d = torch.empty_like(want_d)
        got_d = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                                    w.max_context_len, w.scale, out=got_d, stream=hi)
        done.record(hi)
        main.wait_event(done)
        torch.cuda.synchronize()
        assert torch.equal(got_d, want_d) and torch.equal(got_p, want_p)
    assert pkv.get_device_error() == 0
    G = w.group
    for s in (0, w.num_seqs - 1):
        assert_close(got_d[s, 0:G], oracle_decode_rows(w, s, 0), False, f"seq {s}")
