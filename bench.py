"""Benchmark of one paged-KV attention step on GB300.

Default workload: Llama-2-13B-shaped MHA decode layer (64 sequences, 40/40
heads, head_dim 128, block size 64, context lengths U[128, 4096], bf16 KV,
1.25x pool with permuted page ids).  One step = the append of the batch's new
tokens + paged decode attention over the whole batch, in one call
(pkv_paged_attention_append: planning and append in one launch, split-K
decode, merge); --separate-append makes it two calls (pkv_kv_append, then
pkv_paged_attention).  --workload selects another configuration (1..5).
Configuration 5 is a mixed iteration: one pkv_kv_append of every new row,
then pkv_paged_prefill on the step's stream beside pkv_paged_attention on a
high-priority stream (--mixed-serial: the fused decode call, then the
prefill, on one stream).

Prints ONE JSON line.  `value` = algorithmic bytes of the step / device time
per step, the steps running back to back with no event inside them (K/V
bytes streamed dominate: 2 * head_dim * element size per token and kv head,
plus q, out, block-table entries and the appended rows).  `roofline` is the
dominant call's own rate from a second pass with CUDA events around each
call, and `roofline.back_to_back` the same call timed with its launches
chained.  A workload whose K/V fits in the L2 is flushed before every step.
`e2e` is the same metric through the public API with inputs copied from
pinned host memory and the output copied back inside the timed region.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload.

N > 1 (torchrun): every rank runs an independent replica on its own GPU
(nothing in the step shards across GPUs); value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak); seq-steps/s per layer"
UNIT = "GB/s"
DEFAULT_WORKLOAD = 2


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def _src_hash(name):
    """sha256 prefix of a kernel source with comments and blank space taken
    out, so that editing a comment does not invalidate a capture."""
    path = os.path.join(ROOT, "paged_kv_attention_31_gb300", "csrc", name)
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode("utf-8")).hexdigest()[:12]


def _ncu_traffic(kernel, workload_name):
    """DRAM bytes per launch from profiles/traffic.json (ncu captures), if
    the entry was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    src = {"decode_kernel": "decode.cu", "decode_mma_kernel": "decode_mma.cu",
           "prefill_kernel": "prefill.cu"}[kernel]
    want = _src_hash(src)
    with open(path) as f:
        entries = json.load(f).get("entries", [])
    for e in entries:
        if e["kernel"] == kernel and e["workload"] == workload_name and e["src"] == want:
            return int(e["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler around the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r)
                          if v.lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# oracle CPU baseline (test infrastructure; only this leg touches oracle/)
# ---------------------------------------------------------------------------
def _oracle_sample(w, seqs, gen_device):
    """Host inputs for the oracle on decode sequences `seqs` (all heads):
    pool pages from the seeded generator (on gen_device, bit-identical to
    the host generator), then the oracle's own kv_append of the new tokens."""
    import oracle
    import workloads as W

    P = w.block_size
    pages, tables = [], []
    for s in seqs:
        n = (int(w.context_lens[s]) + P - 1) // P
        tables.append(np.arange(len(pages), len(pages) + n, dtype=np.int32))
        pages.extend(int(p) for p in w.block_tables[s, :n])
    nb = len(pages)
    maxb = max(len(t) for t in tables)
    bt = np.full((len(seqs), maxb), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    dt = np.uint16 if w.kv_dtype == "bf16" else np.uint8
    pools = []
    for c in ("k", "v"):
        src = W.pool_values(w.seed, c, pages, w.num_kv_heads, P, w.head_dim, gen_device)
        pools.append(W.bf16_bits(src))
    kp = np.zeros((nb, w.num_kv_heads, P, w.head_dim), dt)
    vp = np.zeros_like(kp)
    rows = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3).reshape(nb * P, w.num_kv_heads,
                                                                           w.head_dim))
    oracle.kv_append(rows(pools[0]), rows(pools[1]), np.arange(nb * P, dtype=np.int64), kp, vp,
                     w.kv_dtype, w.k_scale, w.v_scale)
    kn, vn = w.kv_new()
    kn, vn = W.bf16_bits(kn), W.bf16_bits(vn)
    slots = w.decode_slot_mapping()
    remap = {p: i for i, p in enumerate(pages)}
    sel = [s for s in seqs if slots[s] >= 0]
    mapped = np.array([remap[int(slots[s]) // P] * P + int(slots[s]) % P for s in sel], np.int64)
    q = W.bf16_bits(w.q_decode())[list(seqs)]
    return dict(q=np.ascontiguousarray(q), kp=kp, vp=vp, bt=bt,
                cl=np.ascontiguousarray(w.context_lens[list(seqs)]),
                kn=np.ascontiguousarray(kn[sel]), vn=np.ascontiguousarray(vn[sel]),
                slots=mapped)


def _oracle_step(w, inp):
    """One oracle step on the sample: kv_append of the new tokens, attention."""
    import oracle
    kp, vp = inp["kp"].copy(), inp["vp"].copy()
    t0 = time.perf_counter()
    oracle.kv_append(inp["kn"], inp["vn"], inp["slots"], kp, vp, w.kv_dtype, w.k_scale,
                     w.v_scale)
    oracle.paged_attention(inp["q"], kp, vp, inp["bt"], inp["cl"], w.scale, w.kv_dtype,
                           w.k_scale, w.v_scale)
    return time.perf_counter() - t0


def _sample_seqs(w, target_s):
    """Sequences (spread over the batch) whose oracle work is about target_s."""
    per_tok_row = 1.15e-6 * w.head_dim / 128         # seconds per (token, q head)
    order = np.random.default_rng(0).permutation(w.num_seqs)
    seqs, est = [], 0.0
    for s in order:
        seqs.append(int(s))
        est += int(w.context_lens[s]) * w.num_q_heads * per_tok_row
        if est >= target_s:
            break
    return sorted(seqs)


def _sample_bytes(w, seqs):
    per_tok = w.num_kv_heads * 2 * w.head_dim * w.elem_bytes
    return int(sum(int(w.context_lens[s]) for s in seqs)) * per_tok


def _oracle_step_threads(w, inp, threads):
    """The same oracle step on `threads` host threads: kv_append on one, then
    the sample's sequences dealt longest first to the least-loaded thread,
    each thread running the oracle's attention on its share (the C oracle
    runs without the interpreter lock).  Returns (seconds, threads used)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cl = inp["cl"]
    groups, load = [[] for _ in range(threads)], [0] * threads
    for i in np.argsort(-cl, kind="stable"):
        g = int(np.argmin(load))
        groups[g].append(int(i))
        load[g] += int(cl[i])
    groups = [np.array(sorted(g), np.int64) for g in groups if g]
    kp, vp = inp["kp"].copy(), inp["vp"].copy()

    def part(g):
        oracle.paged_attention(inp["q"][g], kp, vp, inp["bt"][g], cl[g], w.scale, w.kv_dtype,
                               w.k_scale, w.v_scale)

    with ThreadPoolExecutor(len(groups)) as ex:
        t0 = time.perf_counter()
        oracle.kv_append(inp["kn"], inp["vn"], inp["slots"], kp, vp, w.kv_dtype, w.k_scale,
                         w.v_scale)
        list(ex.map(part, groups))
        dt = time.perf_counter() - t0
    return dt, len(groups)


def cpu_baseline(w, target_s, gen_device):
    """The oracle timed on the host: one thread (the baseline), and the same
    sample spread over every host core."""
    seqs = _sample_seqs(w, target_s)
    inp = _oracle_sample(w, seqs, gen_device)
    dt = _oracle_step(w, inp)
    nbytes = _sample_bytes(w, seqs)
    what = (f"{len(seqs)} of {w.num_seqs} sequences x all {w.num_q_heads} q heads "
            f"({nbytes / 1e6:.1f} MB of KV), fp64 C oracle")
    one = {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{what}, one thread, {dt:.2f} s"}
    dt_all, used = _oracle_step_threads(w, inp, os.cpu_count() or 1)
    allc = {"value": nbytes / dt_all / 1e9, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{what}, sequences spread over {used} threads of "
                      f"{os.cpu_count()} host cores, {dt_all:.2f} s"}
    return one, allc


# ---------------------------------------------------------------------------
def _workload(i, num_seqs=None):
    import workloads as W
    return W.config(i, num_seqs)


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(bytes_per_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s of `world` independent replicas, timed by the slowest."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    w = _workload(args.workload, args.num_seqs)
    _l2_plan(w, args)
    # each step's sample is sized so that the whole run (warm-up and timed
    # steps) takes about 90 s of oracle work at most, whatever --steps is
    seqs = _sample_seqs(w, min(args.ref_sample_s, 90.0 / max(1, args.steps + args.warmup)))
    inp = _oracle_sample(w, seqs, "cpu")
    for _ in range(args.warmup):
        _oracle_step(w, inp)
    times = [_oracle_step(w, inp) for _ in range(args.steps)]
    nbytes = _sample_bytes(w, seqs)
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"each step: {len(seqs)} of {w.num_seqs} sequences x all "
                                       f"{w.num_q_heads} q heads ({nbytes / 1e6:.1f} MB of KV)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def _l2_plan(w, args, dev=None):
    """Decide whether the timed steps flush the L2 and describe it in args.l2_note.

    The working set of one step is the K/V it streams (the decode batch plus
    the prefill sequences' pages); below twice the L2 the step would run from
    cache, so it is flushed before every step.  Returns the L2 size in bytes."""
    l2_bytes = 0
    try:
        import torch
        if torch.cuda.is_available():
            l2_bytes = int(getattr(torch.cuda.get_device_properties(dev or 0), "L2_cache_size", 0))
    except ImportError:
        pass
    l2_bytes = l2_bytes or 129 * 2 ** 20
    per_tok = w.num_kv_heads * 2 * w.head_dim * w.elem_bytes
    working = w.decode_kv_bytes() + int(np.sum(w.prefill_context_lens, dtype=np.int64)) * per_tok
    args.flush = working < 2 * l2_bytes
    args.l2_note = (f"flushed before every step (a {2 * l2_bytes >> 20} MB write, untimed); "
                    f"each step timed on its own: the {working / 2 ** 20:.2f} MB working set "
                    f"fits in the {l2_bytes >> 20} MB L2" if args.flush else
                    f"no flush: each step streams {working / 2 ** 30:.2f} GB of K/V, more than "
                    f"twice the {l2_bytes >> 20} MB L2")
    return l2_bytes


def _config(w, args):
    c = {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
         "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
         "kv_dtype": w.kv_dtype, "max_context_len": w.max_context_len,
         "mean_context_len": float(np.mean(w.context_lens)), "num_blocks": w.num_blocks,
         "partition_tokens": args.partition or "auto",
         "l2": args.l2_note,
         "parallelism": f"replicas x{args.gpus}",
         "launch": "cuda_graph_replay" if args.graph else "eager",
         "step_calls": ("pkv_kv_append, then pkv_paged_attention (high-priority stream) "
                        "beside pkv_paged_prefill" if getattr(args, "concurrent", False) else
                        "pkv_paged_attention_append" if args.fused else
                        "pkv_kv_append + pkv_paged_attention")}
    if w.num_prefill:
        c["prefill_chunks"] = [int(x) for x in w.prefill_chunk_lens]
    return c


def _packed(tensors, device):
    """One uint8 buffer holding `tensors` back to back, each at a 256-byte
    aligned offset (pinned when on the host), and views of it with the
    tensors' dtypes and shapes: (buffer, views)."""
    import torch
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=device, pin_memory=(str(device) == "cpu"))
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return buf, views


# Other workloads measured in the same run as the headline one, each with its
# own step count (timed regions of tens of milliseconds, whatever --steps is).
OTHER_WORKLOADS = ((3, 300), (4, 150), (5, 400), ("mixed_fp8", 400), (1, 400),
                   ("long_prefill", 100))


def _measure(w, a, dev, peaks, peak_kind, world):
    """Time `a.steps` steps of workload w (after `a.warmup` untimed ones) and
    return the report for it: value, rooflines, e2e, clocks."""
    import torch

    import paged_kv_attention_31_gb300 as pkv
    from device_inputs import device_pools, device_step_inputs

    _, rank, local = _dist()
    l2_bytes = _l2_plan(w, a, dev)
    d = device_step_inputs(w, dev)
    kp, vp = device_pools(w, dev)
    B, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    ws_bytes = pkv.paged_attention_workspace_size(B, Hq, w.max_context_len, kp, a.partition,
                                                  w.k_scale, w.v_scale)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    has_prefill = w.num_prefill > 0
    if has_prefill:
        out_p = torch.empty_like(d["q_prefill"])
        max_q = int(w.prefill_chunk_lens.max())
    stream = torch.cuda.current_stream(dev)
    # The mixed step's two attention calls are independent once the step's
    # rows are appended: by default the decode call runs on a high-priority
    # stream beside the prefill, so each fills the SMs the other's tail leaves
    # idle (the append then is its own call, ahead of both).
    a.concurrent = has_prefill and not a.mixed_serial
    if a.concurrent:
        a.fused = False
        hi_s = torch.cuda.Stream(dev, priority=-1)
        ev_app, ev_dec = torch.cuda.Event(), torch.cuda.Event()

    def step(q, k_new, v_new, slots, bt, cl, qp=None, cu=None, pbt=None, pcl=None, ev=None,
             o=None, op=None, decode_only=False):
        o = out if o is None else o
        if a.concurrent and ev is None and not decode_only:
            m = torch.cuda.current_stream(dev)  # the capture stream under --graph
            pkv.kv_append(k_new, v_new, slots, kp, vp, w.k_scale, w.v_scale)
            ev_app.record(m)
            hi_s.wait_event(ev_app)
            pkv.paged_prefill(qp, cu, kp, vp, pbt, pcl, max_q, w.scale,
                              out=out_p if op is None else op, k_scale=w.k_scale,
                              v_scale=w.v_scale)
            pkv.paged_attention(q, kp, vp, bt, cl, w.max_context_len, w.scale, out=o,
                                workspace=ws, k_scale=w.k_scale, v_scale=w.v_scale,
                                partition_tokens=a.partition, stream=hi_s)
            ev_dec.record(hi_s)
            m.wait_event(ev_dec)
            return
        if a.fused:  # the append runs inside the attention call's planning launch
            if ev is not None:
                ev[0].record(stream)
            pkv.paged_attention_append(q, k_new, v_new, slots, kp, vp, bt, cl, w.max_context_len,
                                       w.scale, out=o, workspace=ws, k_scale=w.k_scale,
                                       v_scale=w.v_scale, partition_tokens=a.partition)
        else:
            if not decode_only:  # a decode-only pass times the attention call alone
                pkv.kv_append(k_new, v_new, slots, kp, vp, w.k_scale, w.v_scale)
            if ev is not None:
                ev[0].record(stream)
            pkv.paged_attention(q, kp, vp, bt, cl, w.max_context_len, w.scale, out=o,
                                workspace=ws, k_scale=w.k_scale, v_scale=w.v_scale,
                                partition_tokens=a.partition)
        if ev is not None:
            ev[1].record(stream)
        if has_prefill and not decode_only:
            if ev is not None:
                ev[2].record(stream)
            pkv.paged_prefill(qp, cu, kp, vp, pbt, pcl, max_q, w.scale,
                              out=out_p if op is None else op, k_scale=w.k_scale,
                              v_scale=w.v_scale)
            if ev is not None:
                ev[3].record(stream)

    args_dev = (d["q"], d["k_new"], d["v_new"], d["slots"], d["block_tables"], d["context_lens"])
    if has_prefill:
        args_dev += (d["q_prefill"], d["cu_seqlens_q"], d["prefill_block_tables"],
                     d["prefill_context_lens"])
    for _ in range(a.warmup):
        step(*args_dev)
    torch.cuda.synchronize(dev)
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    graph = None
    if a.graph:
        # the whole step captured once and replayed (per-kernel timing for the
        # roofline then comes from a short eager loop below)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(*args_dev)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(*args_dev)
        for _ in range(a.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)

    # --- timed region: device-resident inputs -------------------------------------
    # The steps run back to back with no event between a step's calls: an
    # event between two launches ends the programmatic launch chain (the next
    # kernel could otherwise start while the previous one drains).  A step
    # whose working set is not well above the L2 would run from cache: then
    # the L2 is flushed (a write of twice its size) before every step,
    # outside the timed spans, and each step is timed on its own.
    flush_buf = None
    if a.flush:
        flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
           for _ in range(a.steps)]
    spans = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
             for _ in range(a.steps)] if a.flush else None
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(a.steps):
        if spans is not None:
            flush_buf.fill_(i & 255)
            spans[i][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(*args_dev)
        if spans is not None:
            spans[i][1].record(stream)
    t_stop.record(stream)
    torch.cuda.synchronize(dev)
    # per-call timing for the rooflines: the same steps again (eager), CUDA
    # events on the launching stream around each call
    for i in range(a.steps):
        if flush_buf is not None:
            flush_buf.fill_(i & 255)
        step(*args_dev, ev=evs[i])
    torch.cuda.synchronize(dev)
    # the mixed step's decode call alone, back to back (its launches chained)
    dec_chain_ms = None
    if has_prefill:
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(a.steps):
            step(*args_dev, decode_only=True)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        dec_chain_ms = c0.elapsed_time(c1) / a.steps
        # and the prefill call alone, back to back (its rows appended above)
        c0.record(stream)
        for i in range(a.steps):
            pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp,
                              d["prefill_block_tables"], d["prefill_context_lens"], max_q,
                              w.scale, out=out_p, k_scale=w.k_scale, v_scale=w.v_scale)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        pf_chain_ms = c0.elapsed_time(c1) / a.steps
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    elapsed_ms = (t_start.elapsed_time(t_stop) if spans is None
                  else float(sum(x.elapsed_time(y) for x, y in spans)))
    attn_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    prefill_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in evs])) if has_prefill else None
    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # --- end to end through the public API from pinned host memory ------------------
    # Every step copies its inputs from pinned host memory and its outputs
    # back.  A step's inputs sit back to back in one pinned staging buffer and
    # its outputs in one device buffer, so each step is one copy in and one
    # copy out.  Copies run on their own streams into double-buffered device
    # inputs and outputs, so step i's copies overlap the kernels of step i - 1
    # (the kernels themselves stay in order on the compute stream: each
    # step's appends precede its attention).
    outs_dev = [out] + ([out_p] if has_prefill else [])
    nbuf = 2
    hbuf, hviews = _packed(args_dev, "cpu")
    for hv, x in zip(hviews, args_dev):
        hv.copy_(x.cpu())
    dsets = [_packed(args_dev, dev) for _ in range(nbuf)]
    osets = [_packed(outs_dev, dev) for _ in range(nbuf)]
    ohost = [_packed(outs_dev, "cpu") for _ in range(nbuf)]
    h2d = hbuf.numel()
    d2h = osets[0][0].numel()
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]      # inputs of set b landed
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]    # kernels done with set b
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]     # outputs of set b copied back

    def run_set(b):
        o = osets[b][1]
        step(*dsets[b][1], o=o[0], op=o[1] if has_prefill else None)

    def e2e_step(i):
        b = i % nbuf
        if i >= nbuf:
            h2d_s.wait_event(ev_done[b])
        with torch.cuda.stream(h2d_s):
            dsets[b][0].copy_(hbuf, non_blocking=True)
        ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        if i >= nbuf:
            stream.wait_event(ev_out[b])
        run_set(b)
        ev_done[b].record(stream)
        d2h_s.wait_event(ev_done[b])
        with torch.cuda.stream(d2h_s):
            ohost[b][0].copy_(osets[b][0], non_blocking=True)
        ev_out[b].record(d2h_s)

    for i in range(min(a.warmup, 3)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if flush_buf is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        for i in range(a.steps):
            e2e_step(i)
        for b in range(nbuf):
            stream.wait_event(ev_out[b])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        last = ohost[(a.steps - 1) % nbuf][1][0]
        e2e_ms = e0.elapsed_time(e1) / a.steps
    else:  # L2 flushed before each step (untimed); copies and kernels in one stream
        e2e_spans = []
        for i in range(a.steps):
            flush_buf.fill_(i & 255)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            dsets[0][0].copy_(hbuf, non_blocking=True)
            run_set(0)
            ohost[0][0].copy_(osets[0][0], non_blocking=True)
            a1.record(stream)
            e2e_spans.append((a0, a1))
        torch.cuda.synchronize(dev)
        last = ohost[0][1][0]
        e2e_ms = float(sum(x.elapsed_time(y) for x, y in e2e_spans)) / a.steps
    if not torch.equal(last, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during the timed region")

    # --- report ----------------------------------------------------------------------
    step_bytes = w.decode_step_bytes()
    ms = elapsed_ms / a.steps
    value = replica_throughput(step_bytes, world, ms)
    attn_bytes = (w.decode_kv_bytes() + 2 * B * Hq * D * 2 +
                  int(np.sum((w.context_lens.astype(np.int64) + w.block_size - 1)
                             // w.block_size)) * 4 + B * 4)
    if a.fused:  # the timed call also scatters the appended rows (all of them:
        # with prefill chunks in the step, their rows too)
        n_app = w.num_append_tokens
        attn_bytes += n_app * w.num_kv_heads * D * (2 * 2 + 2 * w.elem_bytes) + n_app * 8
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    # the same call's time with its launches chained to the previous step's:
    # the step itself when the call is the whole step, else a loop of the
    # decode call alone
    call_chain_ms = dec_chain_ms if has_prefill else ms
    peak = float(peaks["hbm_gbs"])
    # 4 or 8 q heads per kv head at head_dim 128 run on the tensor-core decode
    kname = ("decode_mma_kernel" if D == 128 and w.group in (4, 8) and w.block_size >= 16
             else "decode_kernel")
    launches_per_step = (2 if a.fused else 3) + (1 if has_prefill else 0)
    # append, plan, decode (+ prefill); fused: plan-and-append, decode
    part, max_splits = pkv.paged_attention_plan(B, Hq, w.max_context_len, kp, a.partition,
                                                w.k_scale, w.v_scale)
    splits = max_splits > 1
    launches_per_step += 1 if splits else 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8_e4m3 kv, bf16 q/out",
        "data": "synthetic", "config": _config(w, a),
        # every sequence of the iteration advances one step (prefill chunks too)
        "seq_steps_per_s": world * (B + w.num_prefill) / (ms * 1e-3),
        "frac_of_hbm_peak": value / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": (f"{kname} (pkv_paged_attention_append: plan and append + "
                                "decode + merge)" if a.fused else
                                f"{kname} (pkv_paged_attention: plan + decode + merge)"),
                     "algorithmic_bytes_per_launch": attn_bytes, "ms_per_launch": attn_ms,
                     "timing": "CUDA events around each call (second pass over the steps)",
                     "traffic": _ncu_traffic(kname, w.name),
                     "back_to_back": {
                         "ms_per_launch": call_chain_ms,
                         "achieved": attn_bytes / (call_chain_ms * 1e-3) / 1e9,
                         "frac": attn_bytes / (call_chain_ms * 1e-3) / 1e9 / peak,
                         "timing": ("the decode call alone, launches chained, one event pair "
                                    "around the loop" if has_prefill else
                                    "the timed steps (the step is this call)")}},
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * a.steps,
        "clocks": clock_info,
    }
    if w.num_sharers > 1:  # shared prefix pages counted once above; per sequence here
        line["logical_kv_gbs"] = (w.decode_kv_bytes(unique=False) +
                                  (attn_bytes - w.decode_kv_bytes())) / (attn_ms * 1e-3) / 1e9
    if has_prefill:
        tokens = B + int(np.sum(w.prefill_chunk_lens))
        line["sequences_per_iteration"] = B + w.num_prefill
        line["tokens_per_iteration"] = tokens
        line["tokens_per_s"] = world * tokens / (ms * 1e-3)
        flops = w.prefill_flops()
        tpeak = float(peaks["bf16_tflops"])
        tflops = flops / (prefill_ms * 1e-3) / 1e12
        # the prefill call is the step's dominant kernel here: it takes the
        # top-level roofline, the decode call's moves beside it
        line["decode_roofline"] = line["roofline"]
        line["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": tpeak,
                            "unit": "TFLOP/s", "frac": tflops / tpeak, "peak_kind": peak_kind,
                            "kernel": ("prefill_kernel (pkv_paged_prefill, tcgen05, "
                                       + ("f16 operands from the FP8 pool)"
                                          if w.kv_dtype != "bf16" else "bf16 operands)")),
                            "algorithmic_flops_per_launch": flops, "ms_per_launch": prefill_ms,
                            "timing": "CUDA events around each call (second pass over the steps)",
                            "traffic": _ncu_traffic("prefill_kernel", w.name),
                            "back_to_back": {
                                "ms_per_launch": pf_chain_ms,
                                "achieved": flops / (pf_chain_ms * 1e-3) / 1e12,
                                "frac": flops / (pf_chain_ms * 1e-3) / 1e12 / tpeak,
                                "timing": "the prefill call alone, launches chained, one event "
                                          "pair around the loop"}}
    del kp, vp, d, ws, out
    torch.cuda.empty_cache()
    return line


def _prefill_l2_note(w, dev):
    """How the prefill-only timing relates to the L2: its pages and q."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or 129 * 2 ** 20
    per_tok = w.num_kv_heads * 2 * w.head_dim * w.elem_bytes
    working = (int(np.sum(w.prefill_context_lens, dtype=np.int64)) * per_tok +
               w.num_prefill_tokens * w.num_q_heads * w.head_dim * 2 * 2)
    return (f"no flush: each call reads {working / 2 ** 20:.0f} MB of pages and q and writes its "
            f"output, more than the {l2 >> 20} MB L2 (the call is bound by the tensor cores)"
            if working > l2 else
            f"no flush: the {working / 2 ** 20:.0f} MB working set fits in the {l2 >> 20} MB L2 "
            f"(the call is bound by the tensor cores)")


def _measure_prefill_only(w, a, dev, peaks, peak_kind, world):
    """Chunked prefill alone (its rows appended once, untimed): the prefill
    call timed back to back over a.steps calls, then with events around each
    call; tensor roofline against the bf16 peak."""
    import torch

    import paged_kv_attention_31_gb300 as pkv
    from device_inputs import device_pools, device_step_inputs

    _, _, local = _dist()
    d = device_step_inputs(w, dev)
    kp, vp = device_pools(w, dev)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    max_q = int(w.prefill_chunk_lens.max())
    out_p = torch.empty_like(d["q_prefill"])
    stream = torch.cuda.current_stream(dev)

    def call():
        pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp, d["prefill_block_tables"],
                          d["prefill_context_lens"], max_q, w.scale, out=out_p,
                          k_scale=w.k_scale, v_scale=w.v_scale)

    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(a.steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.steps)]
    for e in evs:
        e[0].record(stream)
        call()
        e[1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    if pkv.get_device_error() != 0:
        raise RuntimeError("device error during the prefill timing")
    chain_ms = max_over_ranks(t0.elapsed_time(t1) / a.steps, dev)
    call_ms = float(np.mean([x.elapsed_time(y) for x, y in evs]))
    flops = w.prefill_flops()
    tpeak = float(peaks["bf16_tflops"])
    value = world * flops / (chain_ms * 1e-3) / 1e12
    line = {
        "value": value, "unit": "TFLOP/s", "ms_per_step": chain_ms, "steps": a.steps,
        "warmup": a.warmup, "higher_is_better": True,
        "config": {"workload": w.name, "prefill_chunks": [int(x) for x in w.prefill_chunk_lens],
                   "prior_context_lens": [int(x) for x in
                                          w.prefill_context_lens - w.prefill_chunk_lens],
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size,
                   "kv_dtype": w.kv_dtype, "step_calls": "pkv_paged_prefill",
                   "l2": _prefill_l2_note(w, dev)},
        "tokens_per_s": world * w.num_prefill_tokens / (chain_ms * 1e-3),
        "roofline": {"bound": "tensor", "achieved": flops / (call_ms * 1e-3) / 1e12,
                     "peak": tpeak, "unit": "TFLOP/s",
                     "frac": flops / (call_ms * 1e-3) / 1e12 / tpeak, "peak_kind": peak_kind,
                     "kernel": "prefill_kernel (pkv_paged_prefill, tcgen05)",
                     "algorithmic_flops_per_launch": flops, "ms_per_launch": call_ms,
                     "timing": "CUDA events around each call",
                     "traffic": _ncu_traffic("prefill_kernel", w.name),
                     "back_to_back": {"ms_per_launch": chain_ms,
                                      "achieved": flops / (chain_ms * 1e-3) / 1e12,
                                      "frac": flops / (chain_ms * 1e-3) / 1e12 / tpeak,
                                      "timing": "the calls back to back, one event pair around "
                                                "the loop"}},
        "gpu_launches": a.steps,
        "clocks": clock_info,
    }
    del kp, vp, d, out_p
    torch.cuda.empty_cache()
    return line


def run_gpu(args):
    import copy

    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = _peaks()
    w = _workload(args.workload, args.num_seqs)
    cpu_line = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.num_seqs > 0:
        cpu_line = cpu_baseline(w, args.cpu_sample_s, dev)
    if w.num_seqs == 0:  # the long prefill: no decode sequences, no CPU decode sample
        line = _measure_prefill_only(w, args, dev, peaks, peak_kind, world)
        line.update({"metric": "paged chunked-prefill attention TFLOP/s (causal-exact flops)",
                     "n_gpus": world, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                     "data": "synthetic"})
        cpu_line = None
    else:
        line = _measure(w, args, dev, peaks, peak_kind, world)
    if cpu_line is not None:
        line["cpu_baseline"], line["cpu_baseline_all_cores"] = cpu_line
    if not args.no_other_workloads and args.num_seqs is None:
        # every other configuration in the same process, each with its own
        # step count: the headline above stays this run's `value`
        others = {}
        for wid, steps in OTHER_WORKLOADS:
            if wid == args.workload:
                continue
            a = copy.copy(args)
            a.steps, a.warmup, a.graph, a.fused, a.mixed_serial = steps, 10, False, True, False
            a.partition = 0
            wo = _workload(wid)
            m = (_measure_prefill_only if wo.num_seqs == 0 else _measure)(
                wo, a, dev, peaks, peak_kind, world)
            m.pop("metric", None)
            others[wo.name] = m
        line["workloads"] = others
        line["gpu_launches"] += sum(m["gpu_launches"] for m in others.values())
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    type=lambda x: int(x) if x.isdigit() else x,
                    choices=[1, 2, 3, 4, 5, "mixed_fp8", "long_prefill"])
    ap.add_argument("--partition", type=int, default=0,
                    help="split-K partition tokens (0 = library's automatic choice)")
    ap.add_argument("--separate-append", dest="fused", action="store_false",
                    help="two calls per decode step (pkv_kv_append, then pkv_paged_attention) "
                         "instead of pkv_paged_attention_append")
    ap.add_argument("--mixed-serial", action="store_true",
                    help="mixed workload: the decode call, then the prefill call, on one stream "
                         "(default: one append of every new row, then the decode call on a "
                         "high-priority stream beside the prefill)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the step in a CUDA graph and time its replays")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="keep only the first N sequences (a smaller case, for profiling)")
    ap.add_argument("--cpu-sample-s", type=float, default=10.0)
    ap.add_argument("--ref-sample-s", type=float, default=0.5,
                    help="oracle seconds per step of --impl reference at most (less when "
                         "steps x that would exceed about 90 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="measure only --workload (by default every other configuration, and "
                         "the long-context prefill, follow in the same run under 'workloads')")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        if args.workload == "long_prefill":
            ap.error("the reference arm times the decode step: pick a workload 1..5")
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
