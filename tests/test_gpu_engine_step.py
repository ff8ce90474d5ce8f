"""Engine steps driven by the native page manager, on the GPU, against the
oracle.

Each step, as an in-flight-batching engine runs it: the native manager
admits, forks (shared prefix pages), appends (slots plus copy-on-write
pairs) and preempts sequences; the device runs pkv_copy_blocks, then
pkv_kv_append, then pkv_paged_attention over the manager's block tables.
The oracle side replays the same operations on the plain-Python manager
model (its tables must equal the native ones), applies the pairs and the
appends to host pools with oracle.copy_blocks / oracle.kv_append, and runs
oracle.paged_attention.  Pools must agree byte for byte after every step;
outputs within the decode tolerances."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_31_gb300 as pkv
from oracle.kv_cache_manager import KVCacheManagerModel
from tests._gpu_state import assert_close
from tests._layout import bf16_from_f32

pytestmark = pytest.mark.gpu


class Engine:
    def __init__(self, N, P, M, Hkv, G, D, kv_dtype, seed):
        self.P, self.M, self.Hkv, self.G, self.D = P, M, Hkv, G, D
        self.kv_dtype = kv_dtype
        self.fp8 = kv_dtype == "fp8_e4m3"
        self.ks, self.vs = (0.0131, 0.0097) if self.fp8 else (1.0, 1.0)
        self.nat = pkv.KVCacheManager(N, P, M)
        self.ref = KVCacheManagerModel(N, P, M)
        dt = np.uint8 if self.fp8 else np.uint16
        self.hk = np.zeros((N, Hkv, P, D), dt)
        self.hv = np.zeros((N, Hkv, P, D), dt)
        tdt = torch.uint8 if self.fp8 else torch.bfloat16
        self.gk = torch.zeros((N, Hkv, P, D), dtype=tdt, device="cuda")
        self.gv = torch.zeros((N, Hkv, P, D), dtype=tdt, device="cuda")
        self.rng = np.random.default_rng(seed)
        self.copies = 0
        self.preempted = 0

    def num_free(self):
        assert self.nat.num_free() == self.ref.num_free()
        return self.nat.num_free()

    def blocks_needed(self, ids, counts):
        return self.both("blocks_needed", ids, counts)

    def preempt_for(self, needed, protected):
        st, victims = self.both("preempt_for", needed, protected)
        self.preempted += len(victims)
        return st, victims

    def both(self, name, *args):
        a = getattr(self.nat, name)(*args)
        b = getattr(self.ref, name)(*args)
        assert a == b, (name, args, a, b)
        return a

    def append(self, ids, counts):
        st, slots, cp = self.nat.append(ids, counts)
        st2, slots2, cp2 = self.ref.append(ids, counts)
        assert st == st2 and np.array_equal(slots, slots2) and np.array_equal(cp, cp2)
        if st != pkv.PKV_OK:
            return st
        T = len(slots)
        self.copies += len(cp)
        kn = bf16_from_f32(self.rng.standard_normal((T, self.Hkv, self.D)).astype(np.float32))
        vn = bf16_from_f32(self.rng.standard_normal((T, self.Hkv, self.D)).astype(np.float32))
        # device: copies first, then the new rows
        pkv.copy_blocks(self.gk, self.gv, torch.from_numpy(cp).cuda(), k_scale=self.ks,
                        v_scale=self.vs)
        to_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        pkv.kv_append(to_bf16(kn), to_bf16(vn), torch.from_numpy(slots).cuda(), self.gk,
                      self.gv, self.ks, self.vs)
        # oracle
        oracle.copy_blocks(self.hk, self.hv, cp)
        oracle.kv_append(kn, vn, slots, self.hk, self.hv, self.kv_dtype, self.ks, self.vs)
        return st

    def check_pools(self):
        assert pkv.get_device_error() == 0
        bits = lambda t: (t.cpu().numpy() if self.fp8 else
                          t.cpu().view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(bits(self.gk), self.hk)
        assert np.array_equal(bits(self.gv), self.hv)

    def attend(self, ids):
        tab, lens = self.nat.block_tables(ids)
        tab2, lens2 = self.ref.block_tables(ids)
        assert np.array_equal(tab, tab2) and np.array_equal(lens, lens2)
        Hq = self.Hkv * self.G
        q = bf16_from_f32(self.rng.standard_normal((len(ids), Hq, self.D)).astype(np.float32))
        scale = 1.0 / np.sqrt(self.D)
        out = pkv.paged_attention(torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16),
                                  self.gk, self.gv, torch.from_numpy(tab).cuda(),
                                  torch.from_numpy(lens).cuda(), int(lens.max()), scale,
                                  k_scale=self.ks, v_scale=self.vs, partition_tokens=2 * self.P)
        assert pkv.get_device_error() == 0
        want = oracle.paged_attention(q, self.hk, self.hv, tab, lens, scale, self.kv_dtype,
                                      self.ks, self.vs)
        assert_close(out, want, self.fp8, f"step over {ids}")


def schedule(e, plan, steps=14):
    """A small in-flight-batching loop: every other step admits a request with
    a short prompt; every step appends one token to each running sequence;
    when the pool is short, running sequences are preempted last in, first
    out (sequence 0 and the request being admitted are protected).  `e`
    needs both/append/blocks_needed/preempt_for/num_free; yields each step's
    running sequences."""
    P = e.P
    e.both("add", 0)
    assert e.append([0], [P + P // 2 + 3]) == pkv.PKV_OK
    e.both("fork", 0, 1, P + P // 2 + 3)     # shares a half-filled page
    e.both("fork", 0, 2, P)                  # page-aligned share
    live, next_id = [0, 1, 2], 3
    yield live
    for step in range(steps):
        if step % 2 == 1:
            new, c = next_id, int(plan.integers(1, 2 * P))
            next_id += 1
            e.both("add", new)
            need = e.blocks_needed([new], [c])
            if need > e.num_free():
                st, victims = e.preempt_for(need, [0, new])
                live = [s for s in live if s not in victims]
            if e.append([new], [c]) == pkv.PKV_OK:
                live.append(new)
            else:
                e.both("release", new)
        need = e.blocks_needed(live, [1] * len(live))
        if need > e.num_free():
            st, victims = e.preempt_for(need, [0])
            live = [s for s in live if s not in victims]
        assert e.append(live, [1] * len(live)) == pkv.PKV_OK
        yield live


@pytest.mark.parametrize("kv_dtype,G,D,P", [("bf16", 4, 128, 16), ("bf16", 2, 64, 32),
                                            ("fp8_e4m3", 8, 128, 16), ("fp8_e4m3", 1, 128, 32)])
def test_engine_steps_with_sharing_copy_on_write_and_preemption(kv_dtype, G, D, P):
    e = Engine(N=12, P=P, M=12, Hkv=2, G=G, D=D, kv_dtype=kv_dtype, seed=7 + G + P)
    for live in schedule(e, np.random.default_rng(100 + P)):
        e.check_pools()
        e.attend(live)
    assert e.copies > 0 and e.preempted > 0        # both paths were exercised


def test_copy_blocks_out_of_range_is_reported_and_skipped():
    e = Engine(N=8, P=16, M=4, Hkv=2, G=4, D=128, kv_dtype="bf16", seed=3)
    e.gk.view(torch.int16).random_(0, 1 << 14)
    e.gv.view(torch.int16).random_(0, 1 << 14)
    before_k, before_v = e.gk.clone(), e.gv.clone()
    pairs = torch.tensor([[0, 5], [1, 99], [-2, 6]], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(e.gk, e.gv, pairs)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    assert torch.equal(e.gk[5].view(torch.int16), before_k[0].view(torch.int16))
    assert torch.equal(e.gv[5].view(torch.int16), before_v[0].view(torch.int16))
    rest = [i for i in range(8) if i != 5]
    assert torch.equal(e.gk[rest].view(torch.int16), before_k[rest].view(torch.int16))
