"""The windowed prefill oracle (rows r0 .. r1-1 of a chunk, run as the last
rows of the sequence cut at L - C + r1) gives exactly the full-chunk
oracle's rows: each row's causal softmax depends only on keys 0 .. its
position.  The full-size long-context parity test relies on it."""
import numpy as np
import pytest

import workloads as W
from tests._gpu_state import oracle_prefill_rows, oracle_prefill_window


@pytest.mark.parametrize("kv_dtype,head_scales", [("bf16", False), ("fp8_e4m3", False),
                                                  ("fp8_e4m3", True)])
def test_window_rows_equal_full_chunk_rows(kv_dtype, head_scales):
    w = W.make_mixed(f"window_{kv_dtype}_{head_scales}", 77, [9], [200, 0], [70, 33], 8, 2, 64,
                     16, kv_dtype=kv_dtype)
    if head_scales:
        w = W.with_head_scales(w)
    kn, vn = w.kv_new()
    for s in range(w.num_prefill):
        C = int(w.prefill_chunk_lens[s])
        for h in range(w.num_kv_heads):
            kv = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
            full = oracle_prefill_rows(w, s, h, kv)
            for r0, r1 in [(0, 1), (0, C), (C // 3, C // 3 + 5), (C - 7, C)]:
                win = oracle_prefill_window(w, s, h, r0, r1, kv)
                assert win.shape == (r1 - r0, w.group, w.head_dim)
                np.testing.assert_array_equal(win, full[r0:r1])
