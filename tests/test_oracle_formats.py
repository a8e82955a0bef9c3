"""Pins of the oracle's format decoders against values fixed outside it."""
import math
import os

import numpy as np
import pytest
import torch

import oracle


def _read_table(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((int(a, 16), float(b)))
    return rows


def test_e4m3_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3fn(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.array_equal(np.signbit(ours[~both_nan]), np.signbit(ref[~both_nan]))
    assert int(np.isnan(ours).sum()) == 2            # only 0x7F and 0xFF


def test_e4m3_landmarks(golden_dir):
    for code, val in _read_table(os.path.join(golden_dir, "e4m3fn_points.txt")):
        got = float(oracle.decode_e4m3fn(np.uint8(code)))
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e2m1_table(golden_dir):
    table = _read_table(os.path.join(golden_dir, "e2m1_ocp.txt"))
    assert len(table) == 16
    for code, val in table:
        got = float(oracle.decode_e2m1(np.uint8(code)))
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e2m1_ignores_high_nibble():
    n = np.arange(256, dtype=np.uint8)
    assert np.array_equal(oracle.decode_e2m1(n), oracle.decode_e2m1(n & 0xF))


def test_bf16_against_torch():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_ue8m0_powers_and_sentinel():
    b = np.arange(256, dtype=np.uint8)
    v = oracle.decode_ue8m0(b)
    assert v[0] == 0.0                         # the page's zero sentinel
    assert v[127] == 1.0 and v[128] == 2.0 and v[126] == 0.5
    assert np.all(v[1:] == np.ldexp(1.0, b[1:].astype(np.int64) - 127))


def test_nibble_order():
    from oracle.formats import unpack_nibbles
    assert unpack_nibbles(np.array([0x21, 0xF0], dtype=np.uint8)).tolist() == [1, 2, 0, 15]


def test_round_e4m3_against_torch_cast():
    # torch's float32 -> float8_e4m3fn cast rounds to nearest even; it has no
    # saturation, so the values are clipped to +-448 first.
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 0.01,
                        rng.uniform(-600, 600, 5000)]).astype(np.float32)
    got = oracle.round_e4m3(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got, ref)


def test_round_e4m3_fixed_points_ties_saturation():
    vals = oracle.decode_e4m3fn(np.arange(256, dtype=np.uint8))
    fin = ~np.isnan(vals)
    assert np.array_equal(oracle.round_e4m3(vals[fin]), vals[fin])          # every code is a fixed point
    # halfway cases of the e4m3fn grid go to the even code
    cases = [(1.0625, 1.0),            # between 1.0 (0x38) and 1.125 (0x39)
             (1.1875, 1.25),           # between 1.125 (0x39) and 1.25 (0x3A)
             (2.0 ** -10, 0.0),        # between 0 and the smallest subnormal 2^-9
             (3 * 2.0 ** -10, 2.0 ** -8),
             (240.0, 240.0), (232.0, 224.0), (248.0, 256.0),
             (-1.0625, -1.0), (460.0, 448.0), (1e9, 448.0), (-1e9, -448.0)]
    for x, want in cases:
        assert float(oracle.round_e4m3(x)) == want, x
    assert np.isnan(oracle.round_e4m3(np.nan))
