"""Pins the oracle's number formats against things other than itself:
numpy/torch conversion routines, the OCP E4M3 definition worked by hand
(tests/golden/e4m3_codes.json), and structural facts (monotonicity, round
trips, symmetry)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse(v: str) -> float:
    v = v.strip()
    if v == "nan":
        return math.nan
    if v in ("inf", "-inf"):
        return math.inf if v == "inf" else -math.inf
    if v == "-0":
        return -0.0
    if "^" in v:
        if "*" in v:
            a, b = v.split("*")
            return float(a) * 2.0 ** float(b.split("^")[1])
        sign = -1.0 if v.startswith("-") else 1.0
        return sign * 2.0 ** float(v.lstrip("-").split("^")[1])
    return float(v)


def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_all_patterns_match_float32_upper_half():
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.bf16_to_double(bits.astype(np.uint16))
    ref = (bits << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # and against torch's bfloat16
    t = torch.from_numpy(bits.astype(np.int32).astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(ours[~nan], t[~nan])


def test_e4m3_decode_golden_values():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code, val in g["decode"].items():
        got = float(oracle.e4m3_to_double(np.array([int(code, 16)], np.uint8))[0])
        want = _parse(val)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_double(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_structure():
    vals = oracle.e4m3_to_double(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(vals) > 0), "non-negative finite codes increase with the code"
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6
    neg = oracle.e4m3_to_double(np.arange(128, 255, dtype=np.uint8))
    assert np.array_equal(neg, -vals)
    # spacing inside a binade is constant: 8 steps per power of two
    for e in range(1, 15):
        b = vals[8 * e: 8 * e + 8]
        assert np.allclose(np.diff(b), b[0] / 8)


def test_e4m3_encode_golden_rows():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for x, code, why in g["encode_rne_satfinite"]:
        got = int(oracle.float_to_e4m3(np.array([_parse(x)], np.float32))[0])
        assert got == int(code, 16), (x, hex(got), code, why)


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_to_double(codes).astype(np.float32)
    assert np.array_equal(oracle.float_to_e4m3(vals), codes)


def test_e4m3_encode_matches_torch_in_range_and_saturates_above():
    rng = np.random.default_rng(0)
    # every bf16 pattern as a float32, plus random float32 values over the range
    bf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    rnd = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 7, 200000))).astype(np.float32)
    # midpoints between neighbouring codes and their float32 neighbours
    pos = oracle.e4m3_to_double(np.arange(127, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    mids = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    y = np.concatenate([bf, rnd, mids, -mids])
    ours = oracle.float_to_e4m3(y)
    ref = torch.from_numpy(y.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    a = np.abs(y)
    inrange = a < 464.0  # torch turns overflow into NaN; below 464 both round to nearest-even
    ok = inrange & ~np.isnan(y)
    assert np.array_equal(ours[ok], ref[ok])
    sat = (a >= 448.0) & ~np.isnan(y)
    assert np.all((ours[sat] & 0x7F) == 0x7E)
    assert np.array_equal(ours[sat] >> 7, np.signbit(y[sat]).astype(np.uint8))
    assert np.all((ours[np.isnan(y)] & 0x7F) == 0x7F)
    # monotone: a larger input never gets a smaller value
    fin = ~np.isnan(y)
    order = np.argsort(y[fin], kind="stable")
    dec = oracle.e4m3_to_double(ours[fin][order])
    assert np.all(np.diff(dec) >= 0)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(300000) * np.exp(rng.uniform(-20, 12, 300000))
    # exact midpoints between f16 neighbours (ties) and values around the overflow edge
    h = np.arange(0, 0x7BFF, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = (h[:-1] + h[1:]) / 2
    x = np.concatenate([x, mid, -mid, [65504.0, 65519.99, 65520.0, 1e6, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26]])
    ours = oracle.round_out(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    # float32-representable inputs, so torch's float32 -> bfloat16 step is the only rounding
    x = (rng.standard_normal(300000) * np.exp(rng.uniform(-80, 80, 300000))).astype(np.float32)
    b = np.arange(0, 0x7F7F, dtype=np.uint32)
    lo = (b << 16).view(np.float32).astype(np.float64)
    hi = ((b + 1) << 16).view(np.float32).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)  # exact in float32
    x = np.concatenate([x, mid, -mid]).astype(np.float32)
    ours = oracle.round_out(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
