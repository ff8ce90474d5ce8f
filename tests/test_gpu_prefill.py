"""Chunked-prefill attention (tcgen05 kernel) on the GPU against the oracle.

Tolerances as for decode: bf16 pools max |err| <= 2e-2, mean |err| <= 2e-3;
FP8 pools max |err| <= 6e-2 against the oracle run on the same stored codes
("TensorRT-LLM框架解析与高性能推理优化实践" §5.3 chunked context over the cache
that §7.2 stores quantised and dequantises inside attention).
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_31_gb300 as pkv
import workloads as W
from tests._gpu_state import (assert_close, device_pools, device_step_inputs,
                              oracle_decode_rows, oracle_prefill_rows, oracle_prefill_window)

pytestmark = pytest.mark.gpu


def _prefill(w, d, kp, vp, append=True):
    ks, vs = w.scale_tensors(d["q_prefill"].device)
    if append:
        pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale,
                      k_scales=ks, v_scales=vs)
    return pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp,
                             d["prefill_block_tables"], d["prefill_context_lens"],
                             int(w.prefill_chunk_lens.max()), w.scale, k_scale=w.k_scale,
                             v_scale=w.v_scale, k_scales=ks, v_scales=vs)


def _check(w, out, seqs=None, heads=None):
    """Rows against the fp64 oracle: bf16 pools at max |err| <= 2e-2 and mean
    <= 2e-3, FP8 pools at max |err| <= 6e-2 (the oracle reads the same codes)."""
    G = w.group
    cu = w.cu_seqlens_q()
    kn, vn = w.kv_new()
    fp8 = w.kv_dtype == "fp8_e4m3"
    for s in (range(w.num_prefill) if seqs is None else seqs):
        for h in (range(w.num_kv_heads) if heads is None else heads):
            kv = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
            want = oracle_prefill_rows(w, s, h, kv)
            assert_close(out[cu[s]:cu[s + 1], h * G:(h + 1) * G], want, fp8,
                         f"{w.name} s={s} h={h}")


def test_small_mixed_config_every_row():
    w = W.small_config(5)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check(w, out)


@pytest.mark.parametrize("G,P", [(1, 16), (2, 32), (4, 32), (8, 64), (4, 16), (16, 64),
                                 (4, 128), (8, 128)])
def test_groups_blocks_and_ragged_chunks(G, P):
    # chunks of 1 token, whole-prompt chunks (prior 0), tails that end
    # mid-tile and mid-key-block
    priors = [0, 7, 64, 129, 0]
    chunks = [1, 33, 200, 64, 257]
    hkv = 2
    w = W.make_mixed(f"prefill_G{G}_P{P}", 900 + G + P, [40], priors, chunks, hkv * G, hkv,
                     128, P)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check(w, out)


@pytest.mark.parametrize("n_chunks", [24, 40])
def test_many_chunks_cta_order(n_chunks):
    # The kernel ranks (sequence, tile pair) groups longest first when there
    # are at most 256 of them (24 chunks x up to 10 pairs) and falls back to a
    # fixed order above that (40 chunks): both must give the same results.
    rng = np.random.default_rng(77 + n_chunks)
    priors = [int(x) for x in rng.integers(0, 600, n_chunks)]
    chunks = [int(x) for x in rng.integers(1, 321, n_chunks)]
    chunks[0] = 320                                   # max_q_len 320: 10 pairs at G = 8
    w = W.make_mixed(f"prefill_many_{n_chunks}", 4242 + n_chunks, [16], priors, chunks, 8, 1,
                     128, 16)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check(w, out, seqs=sorted({0, 1, n_chunks // 2, n_chunks - 1,
                                int(np.argmax(w.prefill_context_lens))}))


@pytest.mark.parametrize("G,P", [(1, 16), (4, 32), (8, 64), (2, 128)])
def test_head_dim_64(G, P):
    priors = [0, 7, 64, 129, 0]
    chunks = [1, 33, 200, 64, 257]
    hkv = 2
    w = W.make_mixed(f"prefill_d64_G{G}_P{P}", 1900 + G + P, [40], priors, chunks, hkv * G, hkv,
                     64, P)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check(w, out)


@pytest.mark.parametrize("D", [128, 64])
def test_zero_length_chunks_in_the_batch(D):
    # sequences with no query tokens this step (equal cu_seqlens entries) sit
    # between real chunks: they own no output rows and disturb no other sequence
    chunks = [64, 0, 129, 0, 1]
    w = W.make_mixed(f"prefill_zero_chunks_d{D}", 5150, [20], [10, 300, 0, 5, 77], chunks,
                     16, 4, D, 32)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    assert out.shape[0] == sum(chunks)
    _check(w, out, seqs=[s for s in range(w.num_prefill) if chunks[s] > 0])


@pytest.mark.parametrize("D,P", [(128, 16), (128, 32), (128, 64), (128, 128), (64, 32), (64, 128)])
def test_never_written_slots_past_the_end_do_not_leak(D, P):
    # fill everything past each sequence's last token with NaN bit patterns;
    # the ends fall inside a page, at a page edge inside a 128-key block and
    # just past a block edge (the last K/V block's tail rows are zeroed before
    # the PV product reads them)
    w = W.make_mixed(f"prefill_nan_tail_D{D}_P{P}", 1234 + D + P, [30], [5, 70, 129, 16],
                     [50, 27, 300, 112], 32, 8, D, P)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    P = w.block_size
    for s in range(w.num_prefill):
        L = int(w.prefill_context_lens[s])
        last = int(w.prefill_block_tables[s, (L - 1) // P])
        off = L % P
        if off:
            kp[last, :, off:, :] = float("nan")
            vp[last, :, off:, :] = float("nan")
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    _check(w, out)


def test_bad_page_id_reported():
    w = W.small_config(5)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    d["prefill_block_tables"] = d["prefill_block_tables"].clone()
    d["prefill_block_tables"][0, 1] = w.num_blocks + 5
    _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS


def test_rows_outside_q_are_reported_and_not_written():
    # the last chunk's end points past num_q_tokens: that sequence is skipped
    # and recorded, the others are computed, nothing lands past the output
    w = W.make_mixed("prefill_bad_cu", 6262, [20], [30, 0, 200], [40, 5, 100], 16, 4, 128, 32)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    T, Hq, D = d["q_prefill"].shape
    big = torch.full((T + 64, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    cu = d["cu_seqlens_q"].clone()
    cu[-1] = T + 40
    pkv.paged_prefill(d["q_prefill"], cu, kp, vp, d["prefill_block_tables"],
                      d["prefill_context_lens"], 200, w.scale, out=big[:T])
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    assert torch.all(big[int(w.cu_seqlens_q()[2]):].float() == 7.0)
    _check(w, big[:T], seqs=[0, 1])


def test_chunk_longer_than_max_q_len_is_reported_and_not_written():
    # max_q_len 32 at G = 4 sizes the grid for one 32-token tile per sequence:
    # the 40- and 100-token chunks are skipped and recorded, the 5-token one runs
    w = W.make_mixed("prefill_short_max_q", 6363, [20], [30, 0, 200], [40, 5, 100], 16, 4, 128,
                     32)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    out = torch.full_like(d["q_prefill"], 7.0)
    pkv.paged_prefill(d["q_prefill"], d["cu_seqlens_q"], kp, vp, d["prefill_block_tables"],
                      d["prefill_context_lens"], 32, w.scale, out=out)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    cu = w.cu_seqlens_q()
    assert torch.all(out[cu[0]:cu[1]].float() == 7.0) and torch.all(out[cu[2]:cu[3]].float() == 7.0)
    _check(w, out, seqs=[1])


def test_full_size_mixed_step_sampled():
    w = W.config(5)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp)
    out_d = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                                w.max_context_len, w.scale)
    out_p = _prefill(w, d, kp, vp, append=False)
    assert pkv.get_device_error() == 0
    G = w.group
    rng = np.random.default_rng(5)
    for s in range(w.num_prefill):
        _check(w, out_p, seqs=[s], heads=[int(rng.integers(0, w.num_kv_heads))])
    for s in (0, int(np.argmax(w.context_lens))):
        h = int(rng.integers(0, w.num_kv_heads))
        assert_close(out_d[s, h * G:(h + 1) * G], oracle_decode_rows(w, s, h), False,
                     f"mixed decode s={s}")


def test_full_size_long_context_prefill_sampled():
    # 8 chunks of 1024 onto prior contexts of 4096 (the benchmark's long-context
    # case): 1024 CTAs in several waves, up to 40 key blocks per tile; 32-row
    # windows at each sampled chunk's start, middle and end against the oracle
    w = W.config("long_prefill")
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    G = w.group
    cu = w.cu_seqlens_q()
    kn, vn = w.kv_new()
    rng = np.random.default_rng(31)
    for s in (0, 3, w.num_prefill - 1):
        h = int(rng.integers(0, w.num_kv_heads))
        kv = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
        C = int(w.prefill_chunk_lens[s])
        for r0 in (0, C // 2 - 16, C - 32):
            want = oracle_prefill_window(w, s, h, r0, r0 + 32, kv)
            assert_close(out[cu[s] + r0:cu[s] + r0 + 32, h * G:(h + 1) * G], want, False,
                         f"{w.name} s={s} h={h} rows {r0}..{r0 + 31}")


# ---- FP8 pools -------------------------------------------------------------------
@pytest.mark.parametrize("G,P,D", [(1, 16, 128), (2, 32, 128), (4, 32, 128), (8, 64, 128),
                                   (16, 64, 128), (4, 128, 128), (8, 16, 64), (2, 128, 64),
                                   (4, 32, 64)])
@pytest.mark.parametrize("head_scales", [False, True])
def test_fp8_pool_groups_blocks_and_ragged_chunks(G, P, D, head_scales):
    priors = [0, 7, 64, 129, 0]
    chunks = [1, 33, 200, 64, 257]
    hkv = 2
    w = W.make_mixed(f"prefill_fp8_G{G}_P{P}_D{D}", 7100 + G + P + D, [40], priors, chunks,
                     hkv * G, hkv, D, P, kv_dtype="fp8_e4m3")
    if head_scales:
        w = W.with_head_scales(w)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    out = _prefill(w, d, kp, vp)
    assert pkv.get_device_error() == 0
    _check(w, out)


def test_fp8_never_written_slots_past_the_end_do_not_leak():
    # E4M3 NaN codes (both signs) in every slot past each sequence's last token
    w = W.make_mixed("prefill_fp8_nan_tail", 7234, [30], [5, 70, 300], [50, 27, 130], 32, 8, 128,
                     32, kv_dtype="fp8_e4m3")
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    P = w.block_size
    for s in range(w.num_prefill):
        L = int(w.prefill_context_lens[s])
        last = int(w.prefill_block_tables[s, (L - 1) // P])
        off = L % P
        if off:
            for pool in (kp, vp):
                pool[last, :, off:, 0::2] = 0x7F
                pool[last, :, off:, 1::2] = 0xFF
    out = _prefill(w, d, kp, vp, append=False)
    assert pkv.get_device_error() == 0
    assert torch.isfinite(out.float()).all()
    _check(w, out)


@pytest.mark.parametrize("mult,scale_div", [(2.0 ** 16, 2.0 ** 16), (2.0 ** -20, 2.0 ** -20),
                                            (300.0, 1.0), (1e-5, 1.0)])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_q_far_from_unit_scale(mult, scale_div, kv_dtype):
    # q rows far outside f16's range (or deep in its subnormals), the softmax
    # scale divided by the same power of two: over an FP8 pool the per-row
    # power-of-two scaling before the f16 conversion keeps the scores exact;
    # over a bf16 pool q is used as it is
    w = W.make_mixed(f"prefill_qrange_{kv_dtype}", 7321, [20], [0, 90], [70, 150], 32, 8, 128,
                     32, kv_dtype=kv_dtype)
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    q_host = (w.q_prefill().float() * mult).to(torch.bfloat16)
    scale = w.scale / scale_div
    out = pkv.paged_prefill(q_host.to("cuda"), d["cu_seqlens_q"], kp, vp,
                            d["prefill_block_tables"], d["prefill_context_lens"],
                            int(w.prefill_chunk_lens.max()), scale, k_scale=w.k_scale,
                            v_scale=w.v_scale)
    assert pkv.get_device_error() == 0
    G = w.group
    cu = w.cu_seqlens_q()
    kn, vn = w.kv_new()
    for s in range(w.num_prefill):
        for h in (0, w.num_kv_heads - 1):
            kv = (W.bf16_bits(kn[:, h, :]), W.bf16_bits(vn[:, h, :]))
            want = _oracle_prefill_rows_q(w, s, h, kv, q_host, scale)
            assert_close(out[cu[s]:cu[s + 1], h * G:(h + 1) * G], want, kv_dtype != "bf16",
                         f"s={s} h={h}")


def _oracle_prefill_rows_q(w, s, h, kv, q_host, scale):
    """oracle_prefill_rows with q and the softmax scale replaced."""
    import oracle
    from tests._gpu_state import host_head_pools
    L, C, P = int(w.prefill_context_lens[s]), int(w.prefill_chunk_lens[s]), w.block_size
    npg = (L + P - 1) // P
    kp, vp = host_head_pools(w, w.prefill_block_tables[s, :npg], h, *kv)
    G = w.group
    cu = w.cu_seqlens_q()
    q = W.bf16_bits(q_host[cu[s]:cu[s + 1], h * G:(h + 1) * G, :])
    ks, vs = w.head_scales(h)
    return oracle.paged_prefill(q, np.array([0, C], np.int32), kp, vp,
                                np.arange(npg, dtype=np.int32)[None], np.array([L], np.int32),
                                scale, w.kv_dtype, ks, vs)


def test_full_size_mixed_step_fp8_sampled():
    w = W.config("mixed_fp8")
    d = device_step_inputs(w)
    kp, vp = device_pools(w)
    pkv.kv_append(d["k_new"], d["v_new"], d["slots"], kp, vp, w.k_scale, w.v_scale)
    out_d = pkv.paged_attention(d["q"], kp, vp, d["block_tables"], d["context_lens"],
                                w.max_context_len, w.scale, k_scale=w.k_scale, v_scale=w.v_scale)
    out_p = _prefill(w, d, kp, vp, append=False)
    assert pkv.get_device_error() == 0
    G = w.group
    rng = np.random.default_rng(6)
    for s in range(w.num_prefill):
        _check(w, out_p, seqs=[s], heads=[int(rng.integers(0, w.num_kv_heads))])
    for s in (0, int(np.argmax(w.context_lens))):
        h = int(rng.integers(0, w.num_kv_heads))
        assert_close(out_d[s, h * G:(h + 1) * G], oracle_decode_rows(w, s, h), True,
                     f"mixed fp8 decode s={s}")
