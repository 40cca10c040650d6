"""Pins for the oracle's element codecs (CPU only).

Each decoder is compared code-by-code with an independent library
conversion (numpy float16, torch bfloat16 / float8_e4m3fn) and with values
the format definitions fix.  The E4M3 encoder is pinned by a brute-force
nearest-value search over the code table (ties to the even code, saturation
to +-448), by torch's own float8 cast on the representable range, and by the
IEEE float32 division the quantiser applies before encoding.
"""
import numpy as np
import pytest
import torch

import oracle


def _same(a, b):
    return np.array_equal(a, b, equal_nan=True)


def test_f16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(codes, oracle.F16)
    want = codes.view(np.float16).astype(np.float64)
    assert _same(got, want)
    # sign of zero preserved
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_bf16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_array(codes, oracle.BF16)
    want = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert _same(got, want)


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_array(codes, oracle.FP8_E4M3)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert _same(got, want)


def test_e4m3_definition_values():
    dec = lambda c: oracle.decode_array(np.array([c], np.uint8), oracle.FP8_E4M3)[0]
    assert dec(0x7E) == 448.0                  # largest finite: 1.75 * 2^8
    assert dec(0x38) == 1.0                    # exponent field 7 = bias
    assert dec(0x08) == 2.0 ** -6              # smallest normal
    assert dec(0x01) == 2.0 ** -9              # smallest subnormal
    assert dec(0x07) == 7 * 2.0 ** -9          # largest subnormal
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0x80) == 0.0 and np.signbit(dec(0x80))
    assert dec(0xFE) == -448.0
    # only the two S.1111.111 codes are NaN: no infinities in E4M3
    vals = oracle.decode_array(np.arange(256, dtype=np.uint8), oracle.FP8_E4M3)
    assert int(np.isnan(vals).sum()) == 2 and not np.isinf(vals).any()


def _table():
    """Finite E4M3 values (from torch, independent of the oracle) -> codes."""
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    pos = [(v, c) for v, c in zip(vals, codes) if np.isfinite(v) and v >= 0 and not (v == 0 and c == 0x80)]
    pos.sort()
    return np.array([v for v, _ in pos]), np.array([c for _, c in pos], dtype=np.uint8)


def _brute_force_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value, ties to the even code, saturating."""
    tv, tc = _table()
    out = np.empty(x.shape, np.uint8)
    a = np.abs(x.astype(np.float64))
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    hi = np.clip(np.searchsorted(tv, a, side="left"), 1, len(tv) - 1)
    lo = hi - 1
    dlo, dhi = a - tv[lo], tv[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (tc[hi] % 2 == 0))
    code = np.where(pick_hi, tc[hi], tc[lo])
    code = np.where(a >= tv[-1], tc[-1], code)       # saturate (and +-inf)
    code = np.where(a <= 0, 0, code)
    out[:] = code | sign
    out[np.isnan(x)] = 0x7F
    return out


def test_e4m3_encoder_strided_bit_patterns():
    # every 4099th float32 bit pattern: ~1M values over the whole float range
    bits = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    got = oracle.encode_e4m3(x)
    want = _brute_force_encode(x)
    assert np.array_equal(got, want)


def test_e4m3_encoder_midpoints_and_neighbours():
    tv, _ = _table()
    mids = (tv[1:] + tv[:-1]) / 2            # exact in float32 (few mantissa bits)
    base = np.concatenate([tv, mids, [448.0, 464.0, 480.0, 1e30, np.inf]]).astype(np.float32)
    xs = [base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(0))]
    x = np.concatenate(xs + [-v for v in xs]).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(x), _brute_force_encode(x))


def test_e4m3_encoder_round_trip_and_saturation():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_array(codes, oracle.FP8_E4M3).astype(np.float32)
    finite = np.isfinite(vals)
    assert np.array_equal(oracle.encode_e4m3(vals[finite]), codes[finite])
    sat = oracle.encode_e4m3(np.array([449.0, 464.0, 1e9, np.inf, -np.inf, -1e9], np.float32))
    assert sat.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.encode_e4m3(np.array([np.nan], np.float32))[0] == 0x7F


def test_e4m3_encoder_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1 << 20, generator=g) * torch.exp(torch.randn(1 << 20, generator=g) * 3)
    x = x.clamp(-448, 448).float()
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e4m3(x.numpy()), want)


def test_e4m3_encoder_divides_in_float32():
    g = np.random.default_rng(6)
    x = g.standard_normal(1 << 16).astype(np.float32) * np.float32(3.0)
    scale = np.float32(np.abs(x).max()) / np.float32(448.0)
    got = oracle.encode_e4m3(x, float(scale))
    want = _brute_force_encode((x / scale).astype(np.float32))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# E5M2 (the second fp8 format the pages name)
# ---------------------------------------------------------------------------
def test_e5m2_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_array(codes, oracle.FP8_E5M2)
    want = torch.from_numpy(codes).view(torch.float8_e5m2).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_e5m2_definition_values():
    d = lambda c: oracle.decode_array(np.array([c], np.uint8), oracle.FP8_E5M2)[0]
    assert d(0x3C) == 1.0                       # exponent 15 = bias
    assert d(0x7B) == 57344.0                   # 1.75 * 2^15, the largest finite
    assert d(0x04) == 2.0 ** -14                # smallest normal
    assert d(0x01) == 2.0 ** -16                # smallest subnormal
    assert d(0x7C) == np.inf and d(0xFC) == -np.inf
    assert all(np.isnan(d(c)) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFF))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))


def _e5m2_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e5m2).double().numpy()
    pos = [(v, c) for v, c in zip(vals, codes) if np.isfinite(v) and v >= 0 and not (v == 0 and c == 0x80)]
    pos.sort()
    return np.array([v for v, _ in pos]), np.array([c for _, c in pos], dtype=np.uint8)


def _brute_force_e5m2(x: np.ndarray) -> np.ndarray:
    """Nearest finite E5M2 value, ties to the even code, saturating."""
    tv, tc = _e5m2_table()
    a = np.abs(x.astype(np.float64))
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    hi = np.clip(np.searchsorted(tv, a, side="left"), 1, len(tv) - 1)
    lo = hi - 1
    dlo, dhi = a - tv[lo], tv[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (tc[hi] % 2 == 0))
    code = np.where(pick_hi, tc[hi], tc[lo])
    code = np.where(a >= tv[-1], tc[-1], code)
    code = np.where(a <= 0, 0, code)
    out = (code | sign).astype(np.uint8)
    out[np.isnan(x)] = 0x7F
    return out


def test_e5m2_encoder_strided_bit_patterns_and_midpoints():
    bits = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    assert np.array_equal(oracle.encode_e5m2(x), _brute_force_e5m2(x))
    tv, _ = _e5m2_table()
    mids = (tv[1:] + tv[:-1]) / 2
    base = np.concatenate([tv, mids, [57344.0, 61440.0, 65536.0, 1e30, np.inf]]).astype(np.float32)
    xs = [base, np.nextafter(base, np.float32(np.inf)), np.nextafter(base, np.float32(0))]
    x = np.concatenate(xs + [-v for v in xs]).astype(np.float32)
    assert np.array_equal(oracle.encode_e5m2(x), _brute_force_e5m2(x))


def test_e5m2_encoder_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(9)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 4)
    x = x[x.abs() < 57344]
    want = x.to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e5m2(x.numpy()), want)
    sat = oracle.encode_e5m2(np.array([57344.0, 61439.0, 61440.0, 1e9, np.inf, -np.inf], np.float32))
    assert sat.tolist() == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB]
