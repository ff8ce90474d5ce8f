"""Device-resident inputs of a workload for the CUDA path (the benchmark and
the GPU tests): pools filled with the seeded generator's values and the
step's per-sequence tensors.  Imports the product library (FP8 pools are
encoded by its own append, exactly as an engine fills them) and the
generators in workloads.py; nothing from the oracle.
"""
import numpy as np
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W


def device_pools(w: W.Workload, device="cuda", gen_device=None):
    """Pools holding the generator's values (FP8: encoded by pkv_kv_append).

    gen_device: where the values are generated (default: on `device`); the
    generator gives the same bits on the host, which suits small workloads
    whose device launches should be the library's own."""
    gen = device if gen_device is None else gen_device
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    if w.kv_dtype == "bf16":
        k = W.fill_pool_(torch.empty(shape, dtype=torch.bfloat16, device=gen), w.seed, "k")
        v = W.fill_pool_(torch.empty(shape, dtype=torch.bfloat16, device=gen), w.seed, "v")
        return k.to(device), v.to(device)
    k = torch.empty(shape, dtype=torch.uint8, device=device)
    v = torch.empty(shape, dtype=torch.uint8, device=device)
    ks, vs = w.scale_tensors(device)
    per_page = w.num_kv_heads * w.block_size * w.head_dim
    chunk = max(1, (1 << 25) // per_page)
    P = w.block_size
    for start in range(0, w.num_blocks, chunk):
        stop = min(w.num_blocks, start + chunk)
        ids = np.arange(start, stop)
        rows = lambda x: x.permute(0, 2, 1, 3).reshape(-1, w.num_kv_heads, w.head_dim).contiguous()
        kn = rows(w.pool_source("k", ids, gen)).to(device)
        vn = rows(w.pool_source("v", ids, gen)).to(device)
        slots = torch.arange(start * P, stop * P, dtype=torch.int64, device=device)
        pkv.kv_append(kn, vn, slots, k, v, w.k_scale, w.v_scale, k_scales=ks, v_scales=vs)
    return k, v


def device_step_inputs(w: W.Workload, device="cuda", gen_device=None):
    """q, this step's new K/V rows and slots, block tables and lengths (and
    the prefill chunks' q, offsets, tables and lengths), on the device;
    values generated on gen_device (default: on `device`)."""
    gen = device if gen_device is None else gen_device
    d = {}
    d["q"] = w.q_decode(gen).to(device)
    d["k_new"], d["v_new"] = (x.to(device) for x in w.kv_new(gen))
    d["slots"] = torch.from_numpy(w.append_slot_mapping()).to(device)
    d["block_tables"] = torch.from_numpy(w.block_tables).to(device)
    d["context_lens"] = torch.from_numpy(w.context_lens).to(device)
    if w.num_prefill:
        d["q_prefill"] = w.q_prefill(gen).to(device)
        d["cu_seqlens_q"] = torch.from_numpy(w.cu_seqlens_q()).to(device)
        d["prefill_block_tables"] = torch.from_numpy(w.prefill_block_tables).to(device)
        d["prefill_context_lens"] = torch.from_numpy(w.prefill_context_lens).to(device)
    return d
