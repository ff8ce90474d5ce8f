"""Each pin of the page-manager model must catch a plausible mistake.

The mistakes are planted in subclasses of the oracle model (on the CPU, in
this file only); the pins of tests/test_oracle_cache_manager.py then run
against the mutant, and at least one of them must fail.  This keeps the
pins honest: a pin set that a broken model also passes proves nothing."""
import numpy as np
import pytest

import tests.test_oracle_cache_manager as pins
from oracle.kv_cache_manager import ERR_INVALID_ARG, ERR_OUT_OF_BLOCKS, OK, KVCacheManagerModel


class NoCopyOnWrite(KVCacheManagerModel):
    """Writes into a shared block in place instead of copying it first."""

    def _plan(self, seq_ids, counts):
        saved = list(self.ref)
        self.ref = [min(r, 1) for r in self.ref]
        try:
            return super()._plan(seq_ids, counts)
        finally:
            self.ref = saved

    def append(self, seq_ids, counts):
        saved = list(self.ref)
        self.ref = [min(r, 1) for r in self.ref]   # every block looks private
        st, slots, copies = super().append(seq_ids, counts)
        for b, r in enumerate(saved):
            if r > 1:
                self.ref[b] = r
        return st, slots, copies


class ForwardReleaseOrder(KVCacheManagerModel):
    """Returns a released sequence's blocks first page first."""

    def release(self, seq_id):
        if seq_id not in self.seqs:
            return ERR_INVALID_ARG
        for b in self.seqs.pop(seq_id)[0]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        return OK


class PreemptOneTooMany(KVCacheManagerModel):
    """Keeps preempting until strictly more than the needed blocks are free."""

    def preempt_for(self, needed, protected=()):
        return super().preempt_for(needed + 1, protected)


class ForkDropsPartialPage(KVCacheManagerModel):
    """A fork shares only the parent's full pages, losing a partial last page."""

    def fork(self, parent, child, num_tokens):
        if parent not in self.seqs or child in self.seqs or child < 0:
            return ERR_INVALID_ARG
        ppages, plen, _ = self.seqs[parent]
        if num_tokens < 0 or num_tokens > plen:
            return ERR_INVALID_ARG
        shared = ppages[:num_tokens // self.P]
        for b in shared:
            self.ref[b] += 1
        self.seqs[child] = [list(shared), num_tokens, self.admitted]
        self.admitted += 1
        return OK


def _pin_calls():
    calls = [(name, ()) for name in (
        "test_hand_worked_append_fork_and_copy_on_write", "test_page_aligned_fork_needs_no_copy",
        "test_two_sharers_append_in_one_call", "test_out_of_blocks_is_atomic",
        "test_invalid_requests_are_refused_without_change",
        "test_lifo_preemption_order_and_protection", "test_preemption_counts_shared_pages_once")]
    calls += [("test_random_operations_read_back_and_conserve", (seed,)) for seed in range(6)]
    return calls


def _failing_pins(monkeypatch, model):
    monkeypatch.setattr(pins, "KVCacheManagerModel", model)
    failed = []
    for name, a in _pin_calls():
        try:
            getattr(pins, name)(*a)
        except (AssertionError, IndexError, KeyError, ValueError):
            failed.append(name)
    return failed


def test_the_model_itself_passes_every_pin(monkeypatch):
    assert _failing_pins(monkeypatch, KVCacheManagerModel) == []


@pytest.mark.parametrize("mutant", [NoCopyOnWrite, ForwardReleaseOrder, PreemptOneTooMany,
                                    ForkDropsPartialPage])
def test_a_planted_mistake_fails_a_pin(monkeypatch, mutant):
    assert _failing_pins(monkeypatch, mutant), f"{mutant.__name__} passed every pin"


# ---- the attention oracle: mistakes planted at its boundary -------------------
# The C oracle is not edited; each mutant wraps oracle.paged_attention so that
# it computes what an oracle with the named mistake would compute, and the
# attention pins (tests/test_oracle_attention.py) run against it.
import oracle  # noqa: E402
import tests.test_oracle_attention as attn_pins  # noqa: E402

_real_attention = oracle.paged_attention


def _scale_ignored(q, kp, vp, bt, cl, scale, *a, **k):
    return _real_attention(q, kp, vp, bt, cl, 1.0, *a, **k)


def _last_token_dropped(q, kp, vp, bt, cl, scale, *a, **k):
    return _real_attention(q, kp, vp, bt, np.maximum(np.asarray(cl) - 1, 0).astype(np.int32),
                           scale, *a, **k)


def _heads_interleaved(q, kp, vp, bt, cl, scale, *a, **k):
    # q head j read against kv head j % Hkv instead of j // G
    Hq, Hkv = q.shape[1], kp.shape[1]
    G = Hq // Hkv
    src = np.array([(j % Hkv) * G + (j // Hkv) for j in range(Hq)])   # a permutation
    q2 = np.empty_like(q)
    q2[:, src] = q
    return _real_attention(q2, kp, vp, bt, cl, scale, *a, **k)[:, src]


def _page_off_by_one(q, kp, vp, bt, cl, scale, *a, **k):
    bt2 = np.asarray(bt).copy()
    bt2[:, :-1] = bt2[:, 1:]                       # page j read from table entry j + 1
    bt2[:, -1] = -1
    bt2 = np.where(bt2 >= 0, bt2, np.where(np.asarray(bt) >= 0, np.asarray(bt), -1))
    return _real_attention(q, kp, vp, bt2.astype(np.int32), cl, scale, *a, **k)


def _fp8_scales_swapped(q, kp, vp, bt, cl, scale, kv_dtype="bf16", k_scale=1.0, v_scale=1.0,
                        *a, **k):
    return _real_attention(q, kp, vp, bt, cl, scale, kv_dtype, v_scale, k_scale, *a, **k)


def _attention_pin_calls():
    calls = [("test_decode_matches_dense_sdpa", p) for p in
             [(8, 2, 16, 4), (4, 4, 8, 2), (6, 1, 32, 8)]]
    calls += [(n, ()) for n in ("test_page_permutation_invariance",
                                "test_uniform_scores_give_mean_of_v",
                                "test_single_token_returns_v0_exactly",
                                "test_dominant_key_selects_its_value",
                                "test_gqa_head_mapping",
                                "test_fp8_pool_matches_dense_dequantised")]
    return calls


def _failing_attention_pins(monkeypatch, impl):
    monkeypatch.setattr(oracle, "paged_attention", impl)
    failed = []
    for name, a in _attention_pin_calls():
        try:
            getattr(attn_pins, name)(*a)
        except AssertionError:
            failed.append(name)
    return failed


def test_the_attention_oracle_itself_passes_these_pins(monkeypatch):
    assert _failing_attention_pins(monkeypatch, _real_attention) == []


@pytest.mark.parametrize("mutant", [_scale_ignored, _last_token_dropped, _heads_interleaved,
                                    _page_off_by_one, _fp8_scales_swapped])
def test_a_planted_attention_mistake_fails_a_pin(monkeypatch, mutant):
    assert _failing_attention_pins(monkeypatch, mutant), f"{mutant.__name__} passed every pin"


# ---- prefill and append oracles -------------------------------------------------
_real_prefill = oracle.paged_prefill
_real_append = oracle.kv_append


def _chunk_lens(cu):
    cu = np.asarray(cu)
    return cu[1:] - cu[:-1]


def _prefill_one_key_more(q, cu, kp, vp, bt, cl, scale, *a, **k):
    # causal window one key too wide (key <= position + 1)
    return _real_prefill(q, cu, kp, vp, bt, (np.asarray(cl) + 1).astype(np.int32), scale, *a, **k)


def _prefill_own_key_masked(q, cu, kp, vp, bt, cl, scale, *a, **k):
    # strict mask (key < position): emulated by positions one lower wherever
    # the sequence has a prior token to attend instead
    cl = np.asarray(cl)
    return _real_prefill(q, cu, kp, vp, bt, np.maximum(cl - 1, _chunk_lens(cu)).astype(np.int32),
                         scale, *a, **k)


def _prefill_head_scales_by_q_head(q, cu, kp, vp, bt, cl, scale, kv_dtype="bf16",
                                   k_scale=1.0, v_scale=1.0, k_scales=None, v_scales=None):
    """Per-head FP8 scales looked up by q head (modulo the kv heads) instead
    of by the q head's kv head."""
    if k_scales is None:
        return _real_prefill(q, cu, kp, vp, bt, cl, scale, kv_dtype, k_scale, v_scale)
    hkv, Hq = kp.shape[1], q.shape[1]
    out = np.zeros(q.shape, np.float64)
    for a in range(Hq):
        out[:, a] = _real_prefill(q[:, [a]], cu, kp[:, [a // (Hq // hkv)]],
                                  vp[:, [a // (Hq // hkv)]], bt, cl, scale, kv_dtype,
                                  float(k_scales[a % hkv]), float(v_scales[a % hkv]))[:, 0]
    return out


def _prefill_fp8_scales_swapped(q, cu, kp, vp, bt, cl, scale, kv_dtype="bf16", k_scale=1.0,
                                v_scale=1.0, k_scales=None, v_scales=None):
    return _real_prefill(q, cu, kp, vp, bt, cl, scale, kv_dtype, v_scale, k_scale,
                         k_scales=v_scales, v_scales=k_scales)


def _append_slot_plus_one(k_new, v_new, slots, kp, vp, *a, **k):
    return _real_append(k_new, v_new, (np.asarray(slots) + 1).astype(np.int64), kp, vp, *a, **k)


def _failing_calls(monkeypatch, attr, impl, calls):
    monkeypatch.setattr(oracle, attr, impl)
    failed = []
    for name, a in calls:
        try:
            getattr(attn_pins, name)(*a)
        except (AssertionError, ValueError, RuntimeError):
            failed.append(name)
    return failed


_PREFILL_PINS = [(n, ()) for n in ("test_prefill_matches_masked_dense_sdpa",
                                   "test_prefill_chunk_of_one_equals_decode",
                                   "test_prefill_row_equals_truncated_decode",
                                   "test_prefill_fp8_row_equals_truncated_decode_with_head_scales")]
_PREFILL_PINS += [("test_prefill_fp8_matches_masked_dense_dequantised", (ph,))
                  for ph in (False, True)]
_APPEND_PINS = [(n, ()) for n in ("test_kv_append_scatter_read_back",
                                  "test_kv_append_out_of_pool_counted_and_skipped",
                                  "test_kv_append_fp8_matches_torch_quantisation",
                                  "test_kv_append_fp8_per_head_scales_match_torch")]


def test_prefill_and_append_oracles_pass_these_pins(monkeypatch):
    assert _failing_calls(monkeypatch, "paged_prefill", _real_prefill, _PREFILL_PINS) == []
    assert _failing_calls(monkeypatch, "kv_append", _real_append, _APPEND_PINS) == []


@pytest.mark.parametrize("mutant", [_prefill_one_key_more, _prefill_own_key_masked,
                                    _prefill_head_scales_by_q_head, _prefill_fp8_scales_swapped])
def test_a_planted_prefill_mistake_fails_a_pin(monkeypatch, mutant):
    assert _failing_calls(monkeypatch, "paged_prefill", mutant, _PREFILL_PINS)


def test_a_planted_append_mistake_fails_a_pin(monkeypatch):
    assert _failing_calls(monkeypatch, "kv_append", _append_slot_plus_one, _APPEND_PINS)
