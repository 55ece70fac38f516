"""Pins for the oracle's scalar number formats (fp16, bf16, OCP e4m3) against
library conversions and the formats' closed forms.  CPU only."""
import numpy as np
import torch


def _structured_f32_sample():
    """Every upper-16-bit pattern of binary32 (sign, exponent, 7 fraction
    bits) with low halves that exercise the rounding bits: exact, just above
    zero, the half-way pattern, just below and above it, all ones."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000],
                    dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    return bits.view(np.float32)


def test_f16_decode_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.f16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_bf16_decode_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_to_f16_rne_matches_numpy(orc):
    x = _structured_f32_sample()
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


def test_f16_rne_ties_and_overflow(orc):
    # 1 + 2^-11 is a tie between 1 and 1+2^-10: goes to even (1.0)
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504, 65519.99, 65520, 2 ** -25,
                  3 * 2 ** -26], dtype=np.float32)
    got = orc.f32_to_f16_bits(x)
    assert got.tolist() == [0x3C00, 0x3C02, 0x7BFF, 0x7BFF, 0x7C00, 0x0000, 0x0001]


def test_e4m3_decode_table(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # closed-form anchors of the format
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_encode_matches_torch_in_range(orc):
    x = _structured_f32_sample()
    x = x[np.isfinite(x) & (np.abs(x) < 448.0)]
    got = orc.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_and_nan(orc):
    x = np.array([448.0, 448.5, 464.0, 1e6, np.inf, -np.inf, -500.0, np.nan, 0.0, -0.0],
                 dtype=np.float32)
    got = orc.f32_to_e4m3(x)
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x00, 0x80]


def test_e4m3_roundtrip_codes(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = orc.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(orc.f32_to_e4m3(vals), codes)


def test_e4m3_ties_to_even(orc):
    # between 1.0 (0x38) and 1.125 (0x39): 1.0625 is a tie -> even mantissa 1.0
    # between 1.125 and 1.25 (0x3A): 1.1875 is a tie -> 1.25
    x = np.array([1.0625, 1.1875, 1.0625 + 2 ** -20, 2 ** -10, 3 * 2 ** -10], np.float32)
    assert orc.f32_to_e4m3(x).tolist() == [0x38, 0x3A, 0x39, 0x00, 0x02]


# ---------------------------------------------------------------- OCP e5m2

def test_e5m2_decode_table(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e5m2_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 6 and all(nan[c] for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # closed-form anchors: infinities, largest finite, one, smallest normal
    # and subnormal
    assert got[0x7C] == np.inf and got[0xFC] == -np.inf
    assert got[0x7B] == 57344.0 and got[0xFB] == -57344.0
    assert got[0x3C] == 1.0 and got[0x04] == 2.0 ** -14 and got[0x01] == 2.0 ** -16


def test_e5m2_encode_matches_torch_in_range(orc):
    x = _structured_f32_sample()
    x = x[np.isfinite(x) & (np.abs(x) < 57344.0)]
    got = orc.f32_to_e5m2(x)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e5m2_encode_saturates_and_nan(orc):
    x = np.array([57344.0, 57344.5, 61440.0, 1e6, np.inf, -np.inf, -60000.0, np.nan, 0.0, -0.0],
                 dtype=np.float32)
    got = orc.f32_to_e5m2(x)
    assert got.tolist() == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0xFB, 0x7F, 0x00, 0x80]


def test_e5m2_roundtrip_codes(orc):
    codes = np.array([c for c in range(256) if (c >> 2) & 0x1F != 31], dtype=np.uint8)
    vals = orc.e5m2_to_f64(codes).astype(np.float32)
    assert np.array_equal(orc.f32_to_e5m2(vals), codes)


def test_e5m2_ties_to_even(orc):
    # 1.125 lies half way between 1.0 (0x3C) and 1.25 (0x3D): even -> 1.0;
    # 1.375 between 1.25 and 1.5 (0x3E): even -> 1.5; in the subnormal
    # range 2^-17 ties to 0 and 3 * 2^-17 to 2 * 2^-16
    x = np.array([1.125, 1.375, 1.125 + 2 ** -20, 2 ** -17, 3 * 2 ** -17], np.float32)
    assert orc.f32_to_e5m2(x).tolist() == [0x3C, 0x3E, 0x3D, 0x00, 0x02]


# ---------------------------------------------------------------- int8 codes

def test_i8_encode_matches_torch_round_and_clamp(orc):
    x = _structured_f32_sample()
    x = x[~np.isnan(x)]
    got = orc.f32_to_i8(x)
    ref = torch.from_numpy(x).round().clamp(-127, 127).to(torch.int8).numpy()
    assert np.array_equal(got, ref)


def test_i8_ties_saturation_nan(orc):
    x = np.array([0.5, 1.5, 2.5, -0.5, -2.5, 126.5, -126.5, 127.0, 127.4, 1e9, np.inf, -np.inf,
                  -200.0, np.nan, -0.0], np.float32)
    assert orc.f32_to_i8(x).tolist() == [0, 2, 2, 0, -2, 126, -126, 127, 127, 127, 127, -127, -127,
                                         0, 0]


def test_i8_symmetric_and_exact_on_integers(orc):
    x = _structured_f32_sample()
    x = x[np.isfinite(x)]
    assert np.array_equal(orc.f32_to_i8(-x), -orc.f32_to_i8(x))
    ints = np.arange(-127, 128, dtype=np.float32)
    assert np.array_equal(orc.f32_to_i8(ints), ints.astype(np.int8))
