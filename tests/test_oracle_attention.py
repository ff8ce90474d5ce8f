"""Pins for the oracle's paged attention, chunked prefill and kv_append.

Each test ties the oracle to something other than itself: torch's SDPA on
dense K/V (brute force), permutation invariance of the physical page order,
closed forms (uniform scores -> mean of V, one token -> V_0, a dominant key),
prefix-shared pages versus private copies, and a read-back of appended slots.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._layout import (bf16_from_f32, bf16_to_f64, dense_attention,
                           paginate)


def _rand_bf16(rng, shape, s=1.0):
    return bf16_from_f32(rng.standard_normal(shape).astype(np.float32) * s)


def _case(seed, lens, Hq, Hkv, D, P, extra_pages=5):
    rng = np.random.default_rng(seed)
    Kd = [_rand_bf16(rng, (L, Hkv, D)) for L in lens]
    Vd = [_rand_bf16(rng, (L, Hkv, D)) for L in lens]
    nb = sum((L + P - 1) // P for L in lens) + extra_pages
    perm_rng = np.random.default_rng(seed + 1)
    kp, bt = paginate(Kd, P, nb, np.random.default_rng(seed + 1))
    vp, bt2 = paginate(Vd, P, nb, np.random.default_rng(seed + 1))
    assert np.array_equal(bt, bt2)
    q = _rand_bf16(rng, (len(lens), Hq, D))
    return q, Kd, Vd, kp, vp, bt, np.array(lens, np.int32)


@pytest.mark.parametrize("Hq,Hkv,D,P", [(8, 2, 16, 4), (4, 4, 8, 2), (6, 1, 32, 8)])
def test_decode_matches_dense_sdpa(Hq, Hkv, D, P):
    lens = [1, 7, 13, 16, 33]
    q, Kd, Vd, kp, vp, bt, cl = _case(10, lens, Hq, Hkv, D, P)
    scale = 1 / math.sqrt(D)
    out = oracle.paged_attention(q, kp, vp, bt, cl, scale)
    for s, L in enumerate(lens):
        ref = dense_attention(bf16_to_f64(q[s])[:, None, :],
                              bf16_to_f64(Kd[s]).transpose(1, 0, 2),
                              bf16_to_f64(Vd[s]).transpose(1, 0, 2), scale)[:, 0, :]
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_page_permutation_invariance():
    lens = [5, 40, 17]
    q, Kd, Vd, kp, vp, bt, cl = _case(11, lens, 4, 2, 16, 4, extra_pages=9)
    out = oracle.paged_attention(q, kp, vp, bt, cl, 0.25)
    rng = np.random.default_rng(99)
    perm = rng.permutation(kp.shape[0])           # new id of old page i
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.paged_attention(q, kp2, vp2, bt2, cl, 0.25)
    assert np.array_equal(out, out2)


def test_uniform_scores_give_mean_of_v():
    lens = [9, 31]
    q, Kd, Vd, kp, vp, bt, cl = _case(12, lens, 4, 2, 16, 4)
    q0 = np.zeros_like(q)                          # all scores equal
    out = oracle.paged_attention(q0, kp, vp, bt, cl, 0.25)
    for s, L in enumerate(lens):
        mean = bf16_to_f64(Vd[s]).mean(axis=0)     # [Hkv, D]
        want = np.repeat(mean, 2, axis=0)          # q head a -> kv head a // 2
        np.testing.assert_allclose(out[s], want, rtol=1e-14, atol=1e-15)


def test_single_token_returns_v0_exactly():
    q, Kd, Vd, kp, vp, bt, cl = _case(13, [1, 1], 8, 4, 16, 4)
    out = oracle.paged_attention(q, kp, vp, bt, cl, 0.25)
    for s in range(2):
        want = np.repeat(bf16_to_f64(Vd[s][0]), 2, axis=0)
        assert np.array_equal(out[s], want)


def test_dominant_key_selects_its_value():
    D, L, P = 16, 37, 8
    rng = np.random.default_rng(14)
    K = np.zeros((L, 1, D), np.float32)
    K[:, 0, 0] = rng.uniform(-1, 1, L)
    K[23, 0, 0] = 64.0                             # score gap > 50 for q = e0
    Kb = bf16_from_f32(K)
    Vb = _rand_bf16(rng, (L, 1, D))
    kp, bt = paginate([Kb], P, 8, np.random.default_rng(1))
    vp, _ = paginate([Vb], P, 8, np.random.default_rng(1))
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    out = oracle.paged_attention(bf16_from_f32(q), kp, vp, bt, np.array([L], np.int32), 1.0)
    np.testing.assert_allclose(out[0, 0], bf16_to_f64(Vb[23, 0]), rtol=0, atol=1e-20)


def test_empty_sequence_gives_zeros():
    q, Kd, Vd, kp, vp, bt, cl = _case(15, [3, 6], 2, 2, 8, 4)
    cl = np.array([0, 6], np.int32)
    out = oracle.paged_attention(q, kp, vp, bt, cl, 0.3)
    assert np.all(out[0] == 0)


def test_prefix_shared_pages_equal_private_copies():
    D, P, Hkv, Hq = 16, 4, 2, 4
    rng = np.random.default_rng(16)
    prefix = 12                                    # 3 whole pages
    Kp = _rand_bf16(rng, (prefix, Hkv, D))
    Vp = _rand_bf16(rng, (prefix, Hkv, D))
    tails = [5, 9]
    Ks = [np.concatenate([Kp, _rand_bf16(rng, (t, Hkv, D))]) for t in tails]
    Vs = [np.concatenate([Vp, _rand_bf16(rng, (t, Hkv, D))]) for t in tails]
    # private copies
    kp, bt = paginate(Ks, P, 20, np.random.default_rng(3))
    vp, _ = paginate(Vs, P, 20, np.random.default_rng(3))
    # shared: point sequence 1's first 3 table entries at sequence 0's pages
    bt_sh = bt.copy()
    bt_sh[1, :3] = bt[0, :3]
    kp_sh = kp.copy()
    vp_sh = vp.copy()
    kp_sh[bt[1, :3]] = 0                           # the private copies are gone
    vp_sh[bt[1, :3]] = 0
    q = _rand_bf16(rng, (2, Hq, D))
    cl = np.array([prefix + t for t in tails], np.int32)
    a = oracle.paged_attention(q, kp, vp, bt, cl, 0.25)
    b = oracle.paged_attention(q, kp_sh, vp_sh, bt_sh, cl, 0.25)
    assert np.array_equal(a, b)


def test_gqa_head_mapping():
    # kv head h holds V == h everywhere; q = 0 -> out[a] = a // G exactly
    D, P, Hkv, G = 8, 4, 4, 3
    L = 10
    K = np.zeros((L, Hkv, D), np.float32)
    V = np.broadcast_to(np.arange(Hkv, dtype=np.float32)[None, :, None], (L, Hkv, D))
    kp, bt = paginate([bf16_from_f32(K)], P, 6, np.random.default_rng(4))
    vp, _ = paginate([bf16_from_f32(V)], P, 6, np.random.default_rng(4))
    q = np.zeros((1, Hkv * G, D), np.uint16)
    out = oracle.paged_attention(q, kp, vp, bt, np.array([L], np.int32), 1.0)
    want = (np.arange(Hkv * G) // G).astype(np.float64)
    assert np.array_equal(out[0, :, 0], want)


def test_fp8_pool_matches_dense_dequantised():
    D, P, Hkv, Hq = 16, 4, 2, 4
    rng = np.random.default_rng(17)
    lens = [6, 19]
    codes = lambda n: rng.integers(0, 256, (n, Hkv, D)).astype(np.uint8)
    Kc = [codes(L) for L in lens]
    Vc = [codes(L) for L in lens]
    for x in Kc + Vc:                              # no NaN codes
        x[(x & 0x7F) == 0x7F] = 0x7E
    kp, bt = paginate(Kc, P, 12, np.random.default_rng(5), np.uint8)
    vp, _ = paginate(Vc, P, 12, np.random.default_rng(5), np.uint8)
    q = _rand_bf16(rng, (2, Hq, D), 0.01)
    ks, vs = 0.011, 0.02
    out = oracle.paged_attention(q, kp, vp, bt, np.array(lens, np.int32), 0.25,
                                 kv_dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
    deq = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for s, L in enumerate(lens):
        ref = dense_attention(bf16_to_f64(q[s])[:, None, :],
                              (deq(Kc[s]) * np.float64(np.float32(ks))).transpose(1, 0, 2),
                              (deq(Vc[s]) * np.float64(np.float32(vs))).transpose(1, 0, 2),
                              0.25)[:, 0, :]
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_bad_page_id_is_reported():
    q, Kd, Vd, kp, vp, bt, cl = _case(18, [5], 2, 2, 8, 4)
    bt = bt.copy()
    bt[0, 1] = kp.shape[0] + 3
    with pytest.raises(ValueError):
        oracle.paged_attention(q, kp, vp, bt, cl, 0.3)


# ---- chunked prefill --------------------------------------------------------
def _prefill_case(seed, priors, chunks, Hq, Hkv, D, P):
    rng = np.random.default_rng(seed)
    lens = [p + c for p, c in zip(priors, chunks)]
    Kd = [_rand_bf16(rng, (L, Hkv, D)) for L in lens]
    Vd = [_rand_bf16(rng, (L, Hkv, D)) for L in lens]
    nb = sum((L + P - 1) // P for L in lens) + 3
    kp, bt = paginate(Kd, P, nb, np.random.default_rng(seed + 1))
    vp, _ = paginate(Vd, P, nb, np.random.default_rng(seed + 1))
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = _rand_bf16(rng, (int(cu[-1]), Hq, D))
    return q, cu, Kd, Vd, kp, vp, bt, np.array(lens, np.int32)


def test_prefill_matches_masked_dense_sdpa():
    priors, chunks = [0, 5, 11], [7, 1, 9]
    Hq, Hkv, D, P = 4, 2, 16, 4
    q, cu, Kd, Vd, kp, vp, bt, cl = _prefill_case(20, priors, chunks, Hq, Hkv, D, P)
    out = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.25)
    for s in range(3):
        L, C = int(cl[s]), chunks[s]
        rows = slice(cu[s], cu[s + 1])
        # bottom-right aligned causal mask: row i sees keys 0 .. L-C+i
        mask = np.arange(L)[None, :] <= (L - C + np.arange(C))[:, None]
        ref = dense_attention(bf16_to_f64(q[rows]).transpose(1, 0, 2),
                              bf16_to_f64(Kd[s]).transpose(1, 0, 2),
                              bf16_to_f64(Vd[s]).transpose(1, 0, 2), 0.25,
                              mask=mask)
        np.testing.assert_allclose(out[rows], ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_prefill_chunk_of_one_equals_decode():
    q, cu, Kd, Vd, kp, vp, bt, cl = _prefill_case(21, [9, 0], [1, 1], 4, 2, 8, 4)
    a = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.5)
    b = oracle.paged_attention(q, kp, vp, bt, cl, 0.5)
    assert np.array_equal(a, b)


def test_prefill_row_equals_truncated_decode():
    q, cu, Kd, Vd, kp, vp, bt, cl = _prefill_case(22, [6], [10], 4, 2, 8, 4)
    out = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.5)
    for i in range(10):
        trunc = np.array([6 + i + 1], np.int32)
        want = oracle.paged_attention(q[i:i + 1], kp, vp, bt, trunc, 0.5)
        assert np.array_equal(out[i], want[0])


def _fp8_prefill_case(seed, priors, chunks, Hq, Hkv, D, P):
    """Pools of random E4M3 codes (NaN codes replaced) and bf16 q."""
    rng = np.random.default_rng(seed)
    lens = [p + c for p, c in zip(priors, chunks)]
    codes = lambda n: rng.integers(0, 256, (n, Hkv, D)).astype(np.uint8)
    Kc = [codes(L) for L in lens]
    Vc = [codes(L) for L in lens]
    for x in Kc + Vc:                              # no NaN codes
        x[(x & 0x7F) == 0x7F] = 0x7E
    nb = sum((L + P - 1) // P for L in lens) + 3
    kp, bt = paginate(Kc, P, nb, np.random.default_rng(seed + 1), np.uint8)
    vp, _ = paginate(Vc, P, nb, np.random.default_rng(seed + 1), np.uint8)
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = _rand_bf16(rng, (int(cu[-1]), Hq, D), 0.05)
    return q, cu, Kc, Vc, kp, vp, bt, np.array(lens, np.int32)


@pytest.mark.parametrize("per_head", [False, True])
def test_prefill_fp8_matches_masked_dense_dequantised(per_head):
    # the chunked prefill over an FP8 pool: torch's E4M3 decoding of the same
    # codes times the scales (per tensor, or per kv head), dense masked SDPA
    priors, chunks = [0, 6, 13], [9, 2, 5]
    Hq, Hkv, D, P = 6, 2, 16, 4
    q, cu, Kc, Vc, kp, vp, bt, cl = _fp8_prefill_case(23, priors, chunks, Hq, Hkv, D, P)
    if per_head:
        ks = np.array([0.011, 0.0045], np.float32)
        vs = np.array([0.02, 0.037], np.float32)
        out = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.25, "fp8_e4m3", 5.0, 5.0,
                                   k_scales=ks, v_scales=vs)
    else:
        ks = np.full(Hkv, 0.011, np.float32)
        vs = np.full(Hkv, 0.02, np.float32)
        out = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.25, "fp8_e4m3", 0.011, 0.02)
    deq = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for s in range(3):
        L, C = int(cl[s]), chunks[s]
        rows = slice(cu[s], cu[s + 1])
        mask = np.arange(L)[None, :] <= (L - C + np.arange(C))[:, None]
        K = deq(Kc[s]) * ks.astype(np.float64)[None, :, None]
        V = deq(Vc[s]) * vs.astype(np.float64)[None, :, None]
        ref = dense_attention(bf16_to_f64(q[rows]).transpose(1, 0, 2), K.transpose(1, 0, 2),
                              V.transpose(1, 0, 2), 0.25, mask=mask)
        np.testing.assert_allclose(out[rows], ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_prefill_fp8_row_equals_truncated_decode_with_head_scales():
    q, cu, Kc, Vc, kp, vp, bt, cl = _fp8_prefill_case(24, [5], [11], 4, 2, 8, 4)
    ks = np.array([0.013, 0.006], np.float32)
    vs = np.array([0.03, 0.011], np.float32)
    out = oracle.paged_prefill(q, cu, kp, vp, bt, cl, 0.5, "fp8_e4m3", k_scales=ks, v_scales=vs)
    for i in range(11):
        trunc = np.array([5 + i + 1], np.int32)
        want = oracle.paged_attention(q[i:i + 1], kp, vp, bt, trunc, 0.5, "fp8_e4m3",
                                      k_scales=ks, v_scales=vs)
        assert np.array_equal(out[i], want[0])


# ---- kv_append ---------------------------------------------------------------
def _slots_view(pool):
    """[num_blocks*P, Hkv, D] view of a pool: row = page*P + offset."""
    nb, hkv, P, D = pool.shape
    return pool.transpose(0, 2, 1, 3).reshape(nb * P, hkv, D)


def test_kv_append_scatter_read_back():
    rng = np.random.default_rng(30)
    nb, hkv, P, D, T = 7, 3, 4, 8, 11
    kp = np.zeros((nb, hkv, P, D), np.uint16)
    vp = np.zeros((nb, hkv, P, D), np.uint16)
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    slots[3] = -1                                  # padding token: skipped
    kn = _rand_bf16(rng, (T, hkv, D))
    vn = _rand_bf16(rng, (T, hkv, D))
    assert oracle.kv_append(kn, vn, slots, kp, vp) == 0
    ks, vs = _slots_view(kp), _slots_view(vp)
    for t in range(T):
        if slots[t] < 0:
            continue
        assert np.array_equal(ks[slots[t]], kn[t])
        assert np.array_equal(vs[slots[t]], vn[t])
    written = np.zeros(nb * P, bool)
    written[slots[slots >= 0]] = True
    assert np.all(ks[~written] == 0) and np.all(vs[~written] == 0)


def test_kv_append_out_of_pool_counted_and_skipped():
    nb, hkv, P, D = 2, 1, 4, 8
    kp = np.zeros((nb, hkv, P, D), np.uint16)
    vp = np.zeros_like(kp)
    kn = np.ones((2, hkv, D), np.uint16)
    assert oracle.kv_append(kn, kn, np.array([nb * P, 1], np.int64), kp, vp) == 1
    assert np.all(_slots_view(kp)[1] == 1) and _slots_view(kp).sum() == D


def test_kv_append_fp8_matches_torch_quantisation():
    rng = np.random.default_rng(31)
    nb, hkv, P, D, T = 5, 2, 4, 16, 9
    kp = np.zeros((nb, hkv, P, D), np.uint8)
    vp = np.zeros_like(kp)
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    kn = _rand_bf16(rng, (T, hkv, D), 2.0)
    vn = _rand_bf16(rng, (T, hkv, D), 0.5)
    ks, vs = np.float32(0.0409), np.float32(0.0093)
    oracle.kv_append(kn, vn, slots, kp, vp, "fp8_e4m3", float(ks), float(vs))
    for new, pool, sc in ((kn, kp, ks), (vn, vp, vs)):
        x = (new.astype(np.uint32) << 16).view(np.float32)
        y = torch.from_numpy(x) / torch.tensor(sc)
        assert float(y.abs().max()) <= 448
        want = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = _slots_view(pool)[slots]
        assert np.array_equal(got, want)


# ---- per-head FP8 scales ("KV Cache量化": one scale per attention head) ----
def test_kv_append_fp8_per_head_scales_match_torch():
    rng = np.random.default_rng(40)
    nb, hkv, P, D, T = 6, 3, 4, 16, 11
    kp = np.zeros((nb, hkv, P, D), np.uint8)
    vp = np.zeros_like(kp)
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    kn = _rand_bf16(rng, (T, hkv, D), 2.0)
    vn = _rand_bf16(rng, (T, hkv, D), 0.5)
    ks = np.array([0.031, 0.0517, 0.09], np.float32)
    vs = np.array([0.0077, 0.0093, 0.021], np.float32)
    oracle.kv_append(kn, vn, slots, kp, vp, "fp8_e4m3", 1.0, 1.0, k_scales=ks, v_scales=vs)
    for new, pool, sc in ((kn, kp, ks), (vn, vp, vs)):
        x = (new.astype(np.uint32) << 16).view(np.float32)          # [T, hkv, D]
        y = torch.from_numpy(x) / torch.from_numpy(sc)[None, :, None]
        assert float(y.abs().max()) <= 448
        want = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(_slots_view(pool)[slots], want)


def test_fp8_per_head_scales_match_dense_dequantised():
    D, P, Hkv, Hq = 16, 4, 2, 6
    rng = np.random.default_rng(41)
    lens = [9, 14]
    codes = lambda n: rng.integers(0, 256, (n, Hkv, D)).astype(np.uint8)
    Kc = [codes(L) for L in lens]
    Vc = [codes(L) for L in lens]
    for x in Kc + Vc:
        x[(x & 0x7F) == 0x7F] = 0x7E
    kp, bt = paginate(Kc, P, 10, np.random.default_rng(6), np.uint8)
    vp, _ = paginate(Vc, P, 10, np.random.default_rng(6), np.uint8)
    q = _rand_bf16(rng, (2, Hq, D), 0.01)
    ks = np.array([0.011, 0.004], np.float32)
    vs = np.array([0.02, 0.05], np.float32)
    out = oracle.paged_attention(q, kp, vp, bt, np.array(lens, np.int32), 0.25,
                                 kv_dtype="fp8_e4m3", k_scales=ks, v_scales=vs)
    deq = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for s, L in enumerate(lens):
        ref = dense_attention(bf16_to_f64(q[s])[:, None, :],
                              (deq(Kc[s]) * ks.astype(np.float64)[None, :, None]).transpose(1, 0, 2),
                              (deq(Vc[s]) * vs.astype(np.float64)[None, :, None]).transpose(1, 0, 2),
                              0.25)[:, 0, :]
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def test_equal_per_head_scales_reduce_to_per_tensor():
    rng = np.random.default_rng(42)
    nb, hkv, P, D, T = 5, 2, 4, 16, 14
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    kn = _rand_bf16(rng, (T, hkv, D))
    vn = _rand_bf16(rng, (T, hkv, D))
    a = [np.zeros((nb, hkv, P, D), np.uint8) for _ in range(4)]
    oracle.kv_append(kn, vn, slots, a[0], a[1], "fp8_e4m3", 0.013, 0.021)
    oracle.kv_append(kn, vn, slots, a[2], a[3], "fp8_e4m3", 9.0, 9.0,
                     k_scales=np.full(hkv, 0.013, np.float32),
                     v_scales=np.full(hkv, 0.021, np.float32))
    assert np.array_equal(a[0], a[2]) and np.array_equal(a[1], a[3])
    bt = np.arange(nb, dtype=np.int32)[None]
    q = _rand_bf16(rng, (1, 4, D))
    cl = np.array([nb * P], np.int32)
    x = oracle.paged_attention(q, a[0], a[1], bt, cl, 0.25, "fp8_e4m3", 0.013, 0.021)
    y = oracle.paged_attention(q, a[0], a[1], bt, cl, 0.25, "fp8_e4m3", 7.0, 7.0,
                               k_scales=np.full(hkv, 0.013, np.float32),
                               v_scales=np.full(hkv, 0.021, np.float32))
    assert np.array_equal(x, y)
