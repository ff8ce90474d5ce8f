"""One prefill chunk and one decode step of two requests through the Python
binding, with the host page manager handing out slots and block tables.
Run it on a machine with a GB300: ``python examples/readme_step.py``."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch
import paged_kv_attention_31_gb300 as pkv

Hq, Hkv, D, P, num_blocks, max_blocks = 32, 8, 128, 32, 1024, 64
k_pool = torch.zeros(num_blocks, Hkv, P, D, dtype=torch.bfloat16, device="cuda")
v_pool = torch.zeros_like(k_pool)
mgr = pkv.KVCacheManager(num_blocks, P, max_blocks)
seqs = [0, 1]
for s in seqs:
    mgr.add(s)

# prefill: a 100-token chunk of each request
status, slots, copies = mgr.append(seqs, [100, 100])
assert status == pkv.PKV_OK
tables, lens = mgr.block_tables(seqs)
bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
k_new = torch.randn(200, Hkv, D, device="cuda").bfloat16()
pkv.kv_append(k_new, torch.randn_like(k_new), torch.from_numpy(slots).cuda(), k_pool, v_pool)
q = torch.randn(200, Hq, D, device="cuda").bfloat16()
cu_seqlens = torch.tensor([0, 100, 200], dtype=torch.int32, device="cuda")
out = pkv.paged_prefill(q, cu_seqlens, k_pool, v_pool, bt, cl, 100, D ** -0.5)

# decode: each request's next token appended and attended in one call
status, slots, copies = mgr.append(seqs, [1, 1])
if len(copies):  # copy-on-write of blocks shared after a fork
    pkv.copy_blocks(k_pool, v_pool, torch.from_numpy(copies).cuda())
tables, lens = mgr.block_tables(seqs)
k_new = torch.randn(2, Hkv, D, device="cuda").bfloat16()
q = torch.randn(2, Hq, D, device="cuda").bfloat16()
out = pkv.paged_attention_append(q, k_new, torch.randn_like(k_new),
                                 torch.from_numpy(slots).cuda(), k_pool, v_pool,
                                 torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                                 int(lens.max()), D ** -0.5)
assert pkv.get_device_error() == 0
print("example ok")
