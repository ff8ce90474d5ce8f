"""The Python binding rejects tensors whose sizes disagree with the call
before anything reaches the library (the C ABI sees only pointers, so a
mismatch there would be an out-of-range device access).  CPU only: the
checks run before any device pointer is taken."""
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv

B, HQ, HKV, D, P, NB, MB = 3, 8, 2, 128, 16, 12, 4


def _args(**over):
    a = dict(q=torch.zeros(B, HQ, D, dtype=torch.bfloat16),
             k_pool=torch.zeros(NB, HKV, P, D, dtype=torch.bfloat16),
             v_pool=torch.zeros(NB, HKV, P, D, dtype=torch.bfloat16),
             block_tables=torch.zeros(B, MB, dtype=torch.int32),
             context_lens=torch.ones(B, dtype=torch.int32))
    a.update(over)
    return a


@pytest.mark.parametrize("bad,msg", [
    (dict(q=torch.zeros(B, HQ, 64, dtype=torch.bfloat16)), "head_dim"),
    (dict(out=torch.zeros(B - 1, HQ, D, dtype=torch.bfloat16)), "out"),
    (dict(out=torch.zeros(B, HQ, D, dtype=torch.float32)), "out"),
    (dict(v_pool=torch.zeros(NB - 1, HKV, P, D, dtype=torch.bfloat16)), "differ"),
    (dict(block_tables=torch.zeros(B - 1, MB, dtype=torch.int32)), "block_tables"),
    (dict(context_lens=torch.ones(B - 1, dtype=torch.int32)), "context_lens"),
])
@pytest.mark.parametrize("fn", ["paged_attention", "paged_attention_noalloc",
                                "paged_attention_append"])
def test_decode_calls_reject_mismatched_sizes(fn, bad, msg):
    a = _args(**{k: v for k, v in bad.items() if k != "out"})
    extra = {"out": bad["out"]} if "out" in bad else {}
    with pytest.raises(ValueError, match=msg):
        if fn == "paged_attention_append":
            kn = torch.zeros(B, HKV, D, dtype=torch.bfloat16)
            pkv.paged_attention_append(a["q"], kn, kn.clone(), torch.zeros(B, dtype=torch.int64),
                                       a["k_pool"], a["v_pool"], a["block_tables"],
                                       a["context_lens"], 64, 0.1, **extra)
        else:
            getattr(pkv, fn)(a["q"], a["k_pool"], a["v_pool"], a["block_tables"],
                             a["context_lens"], 64, 0.1, **extra)


def test_prefill_rejects_mismatched_sizes():
    a = _args()
    q = torch.zeros(10, HQ, D, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4, 10, 10], dtype=torch.int32)
    with pytest.raises(ValueError, match="cu_seqlens_q"):
        pkv.paged_prefill(q, cu[:3], a["k_pool"], a["v_pool"], a["block_tables"],
                          a["context_lens"], 6, 0.1)
    with pytest.raises(ValueError, match="head_dim"):
        pkv.paged_prefill(torch.zeros(10, HQ, 64, dtype=torch.bfloat16), cu, a["k_pool"],
                          a["v_pool"], a["block_tables"], a["context_lens"], 6, 0.1)
    with pytest.raises(ValueError, match="out"):
        pkv.paged_prefill(q, cu, a["k_pool"], a["v_pool"], a["block_tables"], a["context_lens"],
                          6, 0.1, out=torch.zeros(9, HQ, D, dtype=torch.bfloat16))
