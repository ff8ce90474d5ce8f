"""The kernels' failure path on a GPU, without a fault: a bounded wait on a
barrier that nothing arrives at gives up, records PKV_ERR_DEVICE_TIMEOUT and
raises the abort flag (a second wait then returns at once); the kernel ends
normally and the context keeps working: a decode step afterwards is correct."""
import pytest

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import assert_close, device_pools, device_step_inputs, oracle_decode_rows

pytestmark = pytest.mark.gpu


def test_wait_runs_out_is_recorded_and_the_context_stays_usable():
    assert pkv.get_device_error() == 0
    res = pkv.self_test_bounded_wait(2_000_000)   # about 1 ms of SM clocks
    assert res == [0, 0, 1, 1, 1], res
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_TIMEOUT
    assert pkv.get_device_error() == 0            # read and cleared
    w = W.small_config(3)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    out = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                              w.max_context_len, w.scale)
    assert pkv.get_device_error() == 0
    G = w.group
    for s in (0, w.num_seqs - 1):
        assert_close(out[s, 0:G], oracle_decode_rows(w, s, 0), False, f"seq {s}")
