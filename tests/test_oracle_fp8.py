"""Pins for the oracle's E4M3 codec (written from the OCP OFP8 definition).

Independent references: the OCP spec's printed special points (golden file),
torch's own float8_e4m3fn conversion (a separate library implementation), and
closed-form properties of round-to-nearest-even with saturation.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp_points.txt")


def _torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _torch_encode(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_golden_ocp_points():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            code, value = line.split()[:2]
            rows.append((int(code, 16), float(value)))
    assert len(rows) >= 8
    for code, value in rows:
        got = oracle.e4m3_value(np.array([code], np.uint8))[0]
        if math.isnan(value):
            assert math.isnan(got)
            continue
        assert got == value and math.copysign(1, got) == math.copysign(1, value), hex(code)
        assert oracle.e4m3_encode(np.array([value], np.float32))[0] == code


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    ref = _torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign bits agree too (-0 included)
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def _midpoints():
    pos = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    mids = 0.5 * (pos[:-1] + pos[1:])
    return pos, mids


def test_midpoints_round_to_even():
    pos, mids = _midpoints()
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)  # exact in fp32
    got = oracle.e4m3_encode(m32)
    lower = np.arange(0x7E)
    want = np.where(lower % 2 == 0, lower, lower + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    # one ulp either side of each midpoint goes to the nearer neighbour
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    assert np.array_equal(oracle.e4m3_encode(up), (lower + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(dn), lower.astype(np.uint8))


def test_encode_matches_torch_in_range():
    # every bf16 bit pattern whose value lies in [-464, 464] ...
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 464)]
    # ... plus random fp32 values over the whole E4M3 range and the
    # midpoints with their fp32 neighbours
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    rnd = rnd[np.abs(rnd) <= 464]
    _, mids = _midpoints()
    m32 = mids.astype(np.float32)
    x = np.concatenate([vals, rnd, m32, -m32,
                        np.nextafter(m32, np.float32(np.inf)),
                        np.nextafter(m32, np.float32(0))])
    assert np.array_equal(oracle.e4m3_encode(x), _torch_encode(x))


def test_saturation_closed_form():
    # satfinite: anything at or beyond 448 in magnitude (inf included) becomes
    # the largest finite code of the same sign
    x = np.array([448, 464.0001, 465, 480, 1e4, 3e38, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(x) == 0x7E)
    assert np.all(oracle.e4m3_encode(-x) == 0xFE)


def test_quantize_bf16_matches_torch_division_then_cast():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, 20000).astype(np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    ok = np.isfinite(f)
    bits, f = bits[ok], f[ok]
    for scale in (0.010935389436781406, 1.0, 0.37, 3.0e-3):
        s32 = np.float32(scale)
        y = (torch.from_numpy(f) / torch.tensor(s32)).numpy()
        inrange = np.abs(y) <= 464
        want = _torch_encode(y[inrange])
        got = np.array([oracle.quantize_bf16(int(b), float(s32)) for b in bits[inrange][:3000]],
                       np.uint8)
        assert np.array_equal(got, want[:3000])
        assert np.all(np.array([oracle.quantize_bf16(int(b), float(s32))
                                for b in bits[~inrange][:200]]) & 0x7F == 0x7E)
