"""Pins for the oracle's bf16 / e4m3 codecs: the format definitions' fixed
points, exhaustive round trips, tie cases worked by hand, and agreement with
torch's own casts (an independent library implementation)."""

import json
import os

import numpy as np
import pytest
import torch

from oracle import codecs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert int(np.isnan(ours).sum()) == 2          # 0x7F and 0xFF only


def test_e4m3_golden_values():
    with open(os.path.join(GOLDEN, "e4m3_codes.json")) as f:
        g = json.load(f)
    for row in g["decode"]:
        code = int(row["code"], 16)
        v = codecs.e4m3_to_f64(np.array([code], dtype=np.uint8))[0]
        if row["value"] == "nan":
            assert np.isnan(v)
        else:
            assert v == float(row["value"]), row
    for row in g["encode"]:
        c = codecs.f32_to_e4m3(np.array([float(row["x"])], dtype=np.float32))[0]
        assert c == int(row["code"], 16), row


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = codecs.e4m3_to_f64(codes)
    finite = ~np.isnan(vals)
    back = codecs.f32_to_e4m3(vals[finite].astype(np.float32))
    # +0 and -0 are distinct codes and both round-trip
    assert np.array_equal(back, codes[finite])


def test_e4m3_encode_matches_torch_random():
    g = np.random.Generator(np.random.PCG64(7))
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * 50,
        g.standard_normal(50000).astype(np.float32) * 0.01,     # subnormal range
        g.uniform(-448, 448, 50000).astype(np.float32),
    ])
    ours = codecs.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_to_even_every_binade():
    # midpoints between consecutive finite codes round to the even mantissa
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    lo = codecs.e4m3_to_f64(codes)
    hi = codecs.e4m3_to_f64(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo + hi) / 2)   # exact midpoints
    got = codecs.f32_to_e4m3(mid)
    expect = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(got, expect)


def test_e4m3_saturation():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf,
                  -500.0, -np.inf], dtype=np.float32)
    got = codecs.f32_to_e4m3(x)
    assert list(got[:7]) == [0x7E] * 7
    assert list(got[7:]) == [0xFE, 0xFE]
    assert codecs.f32_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_bf16_roundtrip_and_torch():
    g = np.random.Generator(np.random.PCG64(8))
    x = (g.standard_normal(100000) * 10).astype(np.float32)
    ours = codecs.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours, ref)
    back = codecs.bf16_to_f64(ours)
    assert np.array_equal(codecs.f32_to_bf16(back.astype(np.float32)), ours)


def test_bf16_ties():
    # 1 + 2^-8 lies halfway between bf16 1.0 and 1 + 2^-7: ties to even (1.0)
    one = np.float32(1.0)
    x = np.array([one + np.float32(2.0 ** -8), one + np.float32(3 * 2.0 ** -8)], np.float32)
    got = codecs.bf16_to_f64(codecs.f32_to_bf16(x))
    assert got[0] == 1.0
    assert got[1] == 1.0 + 2.0 ** -6       # 1+3*2^-8 is halfway 1+2^-7 / 1+2^-6 -> even


@pytest.mark.parametrize("v", [0.0, -0.0, 1.0, -2.5, 3.0e38])
def test_bf16_exact_values(v):
    b = codecs.f32_to_bf16(np.array([v], np.float32))
    assert codecs.bf16_to_f64(b)[0] == np.float32(v).astype(np.float64) or v == 3.0e38
