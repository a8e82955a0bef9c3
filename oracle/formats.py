"""Decoders of the stored number formats, written from their bit definitions.

TEST INFRASTRUCTURE (see the package header).

* e4m3fn (OCP FP8): sign bit, 4-bit exponent with bias 7, 3-bit mantissa,
  subnormals at exponent 0, S.1111.111 is NaN and there is no infinity.
  [PA] "FNUZ vs OCP" commit: gfx950 reads the fp8 MFMA operands as OCP
  e4m3fn, the format this library stores.
* e2m1 (OCP FP4): sign bit, 2-bit exponent with bias 1, 1-bit mantissa,
  subnormal at exponent 0; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. [UQ] STEP F
  (K codes are e2m1) and [IDX] ``dequant_tile`` (NVFP4 key codes).
* UE8M0: the byte b is the power 2^(b-127); [UQ] STEP F decodes b=0 to +0.
* bf16: the upper 16 bits of an IEEE binary32.

Encoder: ``round_e4m3`` rounds to the nearest e4m3fn value, ties to the
even code, saturating at +-448.

Pins: all 256 e4m3 codes against torch's float8_e4m3fn (and the encoder
against torch's round-to-nearest-even cast, its fixed points and ties); all 16 e2m1 codes
against the OCP value table in tests/golden; bf16 against torch.bfloat16;
UE8M0 against powers of two and the zero sentinel.
"""
import numpy as np


def decode_e4m3fn(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 0x7
    mag = np.where(exp == 0,
                   (man / 8.0) * 2.0 ** (1 - 7),
                   (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0))
    mag = np.where((exp == 0xF) & (man == 0x7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def round_e4m3(x) -> np.ndarray:
    """Values -> nearest e4m3fn value (round to nearest, ties to the even
    code), saturating to +-448; NaN stays NaN. Used for the [UQ] STEP B'
    query haircut (cvt_pk_fp8_f32 of q_r / sqrt(D))."""
    x = np.asarray(x, dtype=np.float64)
    vals = decode_e4m3fn(np.arange(256, dtype=np.uint8))
    pos = np.arange(0, 0x7F)                       # codes 0x00..0x7E: 0 .. 448, increasing
    grid = vals[pos]
    a = np.minimum(np.abs(x), 448.0)
    i = np.clip(np.searchsorted(grid, a), 1, len(grid) - 1)   # grid[i-1] <= a <= grid[i] (a > 0)
    lo, hi = grid[i - 1], grid[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((pos[i] & 1) == 0))
    mag = np.where(a == 0, 0.0, np.where(pick_hi, hi, lo))
    out = np.where(np.signbit(x), -mag, mag)
    return np.where(np.isnan(x), np.nan, out)


def decode_e2m1(nibbles) -> np.ndarray:
    n = np.asarray(nibbles, dtype=np.uint8).astype(np.int64) & 0xF
    sign = (n >> 3) & 1
    exp = (n >> 1) & 0x3
    man = n & 0x1
    mag = np.where(exp == 0,
                   (man / 2.0) * 2.0 ** (1 - 1),
                   (1.0 + man / 2.0) * np.exp2(exp.astype(np.float64) - 1.0))
    return np.where(sign == 1, -mag, mag)


def decode_ue8m0(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8).astype(np.float64)
    return np.where(b == 0, 0.0, np.exp2(b - 127.0))


def decode_bf16(bits) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def unpack_nibbles(packed) -> np.ndarray:
    """[..., n] bytes -> [..., 2n] nibbles; element 2i is the low nibble of
    byte i ([UQ] STEP F stores codes in natural contiguous order; the V
    convert reads byte s as elements 2s and 2s+1)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
