"""Pins of the oracle's bfloat16 and E4M3 codecs against facts outside the oracle:
exhaustive round trips over every bit pattern, torch's own conversions (a library
routine) on the ranges where they define the same rounding, and hand-checked
ties, saturation and signed zeros."""
import numpy as np
import pytest
import torch

from oracle.formats import (bf16_decode, bf16_encode, e4m3_decode, e4m3_encode_sat,
                            e4m3_ordinal, E4M3_MAX)


def test_bf16_decode_matches_binary32_upper_half():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        via_f32 = (bits << 16).view(np.float32).astype(np.float64)
    dec = bf16_decode(bits.astype(np.uint16))
    nan = np.isnan(via_f32)
    assert np.array_equal(np.isnan(dec), nan)
    assert np.array_equal(dec[~nan], via_f32[~nan])


def test_bf16_roundtrip_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    val = bf16_decode(bits)
    ok = ~np.isnan(val)
    assert np.array_equal(bf16_encode(val[ok]), bits[ok])


def test_bf16_encode_matches_torch_on_binary32_inputs():
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    # add subnormals, values near the overflow threshold and exact midpoints
    extra = np.array([1e-40, -3e-41, 3.3895e38, -3.3895e38, 3.39e38, 3.4e38, -3.4e38, 1.00390625, 1.01171875,
                      -1.00390625, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134], np.float32)
    f = np.concatenate([f, extra])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = bf16_encode(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_ties_to_even_hand_checked():
    # 1 + 2^-8 is halfway between 1 (0x3F80) and 1 + 2^-7 (0x3F81): even -> 0x3F80.
    # 1 + 3*2^-8 is halfway between 0x3F81 and 0x3F82: even -> 0x3F82.
    assert bf16_encode(1.0 + 2.0 ** -8) == 0x3F80
    assert bf16_encode(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert bf16_encode(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert bf16_encode(-0.0) == 0x8000
    assert bf16_encode(np.inf) == 0x7F80
    # (2 - 2^-8) * 2^127 is halfway between the largest finite bf16 and 2^128: rounds to inf
    assert bf16_encode((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    assert bf16_encode((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert bf16_encode(1e300) == 0x7F80 and bf16_encode(-2.0 ** 200) == 0xFF80


def test_e4m3_every_finite_code_roundtrips():
    codes = np.arange(256, dtype=np.uint8)
    val = e4m3_decode(codes)
    ok = ~np.isnan(val)
    assert ok.sum() == 254                      # only S.1111.111 are NaN
    assert np.array_equal(e4m3_encode_sat(val[ok]), codes[ok])
    assert np.nanmax(val) == 448.0 and np.nanmin(val) == -448.0
    assert e4m3_decode(np.uint8(1)) == 2.0 ** -9


@pytest.mark.parametrize("scale", [1.0, 0.25, 2.0])
def test_e4m3_codes_roundtrip_through_a_scale(scale):
    """Exactly representable values survive quantise(v*s / s) for power-of-two s
    (spec fact: FP8 codes of exactly representable values round-trip)."""
    from oracle.ops import quant_e4m3_static
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    val = e4m3_decode(codes)
    assert np.array_equal(quant_e4m3_static(val * scale, scale), codes)


def test_e4m3_matches_torch_inside_the_finite_range():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 50, 100_000), rng.normal(0, 0.01, 50_000),
                        rng.uniform(-448, 448, 50_000)]).astype(np.float32)
    # all E4M3 midpoints (ties) between neighbouring finite codes
    pos = np.sort(e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    v = v[np.abs(v) <= 448]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode_sat(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_e4m3_ties_saturation_zero_hand_checked():
    assert e4m3_encode_sat(1.0625) == 0x38       # between 1 and 1.125: even mantissa 0
    assert e4m3_encode_sat(1.1875) == 0x3A       # between 1.125 and 1.25: even mantissa 2
    assert e4m3_encode_sat(464.0) == 0x7E        # beyond 448 saturates, never NaN
    assert e4m3_encode_sat(1e9) == 0x7E
    assert e4m3_encode_sat(-1e9) == 0xFE
    assert e4m3_encode_sat(2.0 ** -10) == 0x00   # half of the smallest subnormal: tie to 0
    assert e4m3_encode_sat(2.0 ** -10 * 1.01) == 0x01
    assert e4m3_encode_sat(-0.0) == 0x80
    assert e4m3_encode_sat(-2.0 ** -11) == 0x80
    assert e4m3_encode_sat(np.nan) == 0x7F
    assert E4M3_MAX == 448.0


def test_e4m3_ordinal_is_monotone_with_adjacent_zeros():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    val = e4m3_decode(codes)
    order = np.lexsort((-(codes >> 7).astype(np.int64), val))   # -0 before +0
    ords = e4m3_ordinal(codes[order])
    assert np.array_equal(np.diff(ords), np.ones(len(ords) - 1, np.int64))
    assert e4m3_ordinal(np.uint8(0x00)) - e4m3_ordinal(np.uint8(0x80)) == 1
