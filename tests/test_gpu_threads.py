"""Several host threads make their first library calls at the same time (in
a fresh process, so the per-device set-up runs concurrently), each on its own
stream and buffers; every result equals the one-thread result bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import device_pools, device_step_inputs

torch.cuda.init()
w5 = W.small_config(5)
w4 = W.small_config(4)
d5, (k5, v5) = device_step_inputs(w5), device_pools(w5)
d4, (k4, v4) = device_step_inputs(w4), device_pools(w4)
torch.cuda.synchronize()
barrier = threading.Barrier(6)
results, errors = {}, []

def decode(w, d, kp, vp, stream):
    return pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                               w.max_context_len, w.scale, k_scale=w.k_scale,
                               v_scale=w.v_scale, stream=stream)

def prefill(w, d, kp, vp, stream):
    return pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp,
                             d["prefill_block_tables"], d["prefill_context_lens"],
                             int(w.prefill_chunk_lens.max()), w.scale, stream=stream)

jobs = [("d5", decode, (w5, d5, k5, v5)), ("p5", prefill, (w5, d5, k5, v5)),
        ("d4", decode, (w4, d4, k4, v4))] * 2

def run(i, name, fn, a):
    try:
        s = torch.cuda.Stream()
        barrier.wait()
        with torch.cuda.stream(s):
            out = fn(*a, stream=s)
        s.synchronize()
        results[i] = (name, out)
    except Exception as e:  # reported to the parent
        errors.append(repr(e))

ts = [threading.Thread(target=run, args=(i,) + j) for i, j in enumerate(jobs)]
for t in ts: t.start()
for t in ts: t.join()
assert not errors, errors
torch.cuda.synchronize()
ref = {"d5": decode(w5, d5, k5, v5, None), "p5": prefill(w5, d5, k5, v5, None),
       "d4": decode(w4, d4, k4, v4, None)}
torch.cuda.synchronize()
for i, (name, out) in results.items():
    assert torch.equal(out, ref[name]), name
assert pkv.get_device_error() == 0
print("ok", len(results))
"""


def test_first_calls_from_several_threads():
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().endswith("ok 6")
