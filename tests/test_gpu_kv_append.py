"""kv_append on the GPU: bit-exact against the oracle's scatter / E4M3 encoder."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_31_gb300 as pkv
from tests._layout import bf16_from_f32

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.cpu().numpy()


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("hkv,P,D", [(8, 32, 128), (3, 16, 64), (1, 64, 128), (2, 128, 128)])
def test_kv_append_bit_exact(fp8, hkv, P, D):
    rng = np.random.default_rng(100 + hkv + P)
    nb, T = 37, 509
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    slots[::17] = -1                                   # padding tokens
    kn = bf16_from_f32(rng.standard_normal((T, hkv, D)).astype(np.float32) * 1.7)
    vn = bf16_from_f32(rng.standard_normal((T, hkv, D)).astype(np.float32) * 0.6)
    dt = np.uint8 if fp8 else np.uint16
    init = rng.integers(0, 120, (nb, hkv, P, D)).astype(dt)   # finite junk
    kp, vp = init.copy(), init.copy()
    ks, vs = (0.02137, 0.00731) if fp8 else (1.0, 1.0)
    oracle.kv_append(kn, vn, slots, kp, vp, "fp8_e4m3" if fp8 else "bf16", ks, vs)

    tdt = torch.uint8 if fp8 else torch.bfloat16
    to_dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    gk = to_dev(init).view(tdt).clone()
    gv = to_dev(init).view(tdt).clone()
    pkv.kv_append(to_dev(kn).view(torch.bfloat16), to_dev(vn).view(torch.bfloat16),
                  torch.from_numpy(slots).cuda(), gk, gv, ks, vs)
    assert pkv.get_device_error() == 0
    assert np.array_equal(_bits(gk), kp)
    assert np.array_equal(_bits(gv), vp)


@pytest.mark.parametrize("hkv,P,D", [(8, 32, 128), (3, 16, 64)])
def test_kv_append_per_head_scales_bit_exact(hkv, P, D):
    # FP8 with one K and one V scale per kv head: head h must be divided by
    # its own scale (a head-index mix-up changes the codes of every token)
    rng = np.random.default_rng(400 + hkv)
    nb, T = 29, 401
    slots = rng.choice(nb * P, T, replace=False).astype(np.int64)
    slots[::13] = -1
    kn = bf16_from_f32(rng.standard_normal((T, hkv, D)).astype(np.float32) * 1.7)
    vn = bf16_from_f32(rng.standard_normal((T, hkv, D)).astype(np.float32) * 0.6)
    ks = (0.011 * (1.0 + 0.61 * np.arange(hkv))).astype(np.float32)
    vs = (0.004 * (1.0 + 0.29 * np.arange(hkv))[::-1]).astype(np.float32)
    init = rng.integers(0, 120, (nb, hkv, P, D)).astype(np.uint8)
    kp, vp = init.copy(), init.copy()
    # the scalar scales are deliberately wrong: the arrays must win
    oracle.kv_append(kn, vn, slots, kp, vp, "fp8_e4m3", 9.0, 9.0, k_scales=ks, v_scales=vs)

    to_dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    gk, gv = to_dev(init).clone(), to_dev(init).clone()
    pkv.kv_append(to_dev(kn).view(torch.bfloat16), to_dev(vn).view(torch.bfloat16),
                  torch.from_numpy(slots).cuda(), gk, gv, 9.0, 9.0,
                  k_scales=torch.from_numpy(ks).cuda(), v_scales=torch.from_numpy(vs).cuda())
    assert pkv.get_device_error() == 0
    assert np.array_equal(_bits(gk), kp)
    assert np.array_equal(_bits(gv), vp)


def test_fp8_encoder_special_values():
    # saturation, ties, subnormals, signed zeros, every bf16 pattern in range
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    keep = np.isfinite(f)
    x = bits[keep].astype(np.uint16)
    D = 128
    T = (len(x) + D - 1) // D
    x = np.concatenate([x, np.zeros(T * D - len(x), np.uint16)]).reshape(T, 1, D)
    for scale in (1.0, 0.0625, 0.010935389, 3.3):
        slots = np.arange(T, dtype=np.int64)
        nb = (T + 15) // 16
        kp = np.zeros((nb, 1, 16, D), np.uint8)
        vp = np.zeros_like(kp)
        oracle.kv_append(x, x, slots, kp, vp, "fp8_e4m3", scale, scale)
        gk = torch.zeros((nb, 1, 16, D), dtype=torch.uint8, device="cuda")
        gv = torch.zeros_like(gk)
        xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        pkv.kv_append(xd, xd, torch.from_numpy(slots).cuda(), gk, gv, scale, scale)
        assert np.array_equal(gk.cpu().numpy(), kp), f"scale {scale}"


def test_out_of_pool_slot_is_reported_and_skipped():
    nb, hkv, P, D = 4, 2, 16, 64
    kp = torch.zeros((nb, hkv, P, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kn = torch.ones((3, hkv, D), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([5, nb * P + 3, 7], dtype=torch.int64, device="cuda")
    assert pkv.get_device_error() == 0
    pkv.kv_append(kn, kn, slots, kp, vp)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_BOUNDS
    rows = kp.permute(0, 2, 1, 3).reshape(nb * P, hkv, D)
    assert rows[5].float().eq(1).all() and rows[7].float().eq(1).all()
    assert rows.float().sum().item() == 2 * hkv * D
    assert pkv.get_device_error() == 0                 # cleared by the read


def test_zero_tokens_is_a_noop():
    kp = torch.zeros((2, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    pkv.kv_append(e, e, torch.empty(0, dtype=torch.int64, device="cuda"), kp, kp.clone())
    assert kp.float().abs().sum().item() == 0
