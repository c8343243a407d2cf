"""Pins for the oracle's FP8 E4M3 page codec (the compressed DRAM tier):
code values from the format definition, round-to-nearest-even on constructed
midpoints, agreement with torch's float8_e4m3fn conversion on random values,
round trips of representable values, the per-row scale, and the error bound of
the codec (3 mantissa bits: half an ulp = 2^-4 relative for normal values).

CPU only; no GPU, no CUDA library."""

import numpy as np
import pytest
import torch

import oracle as O


def test_code_values_from_format():
    v = O.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0            # largest finite
    assert v[0x38] == 1.0 and v[0x08] == 2.0 ** -6          # bias 7, smallest normal
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9  # subnormals
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    finite = v[~np.isnan(v)]
    assert len(finite) == 254 and len(np.unique(finite)) == 253  # +0 and -0 compare equal


def test_round_to_nearest_even_midpoints():
    v = O.e4m3_values()
    cases = {1.0625: 1.0, 1.1875: 1.25, 2.0 ** -10: 0.0, 1.5 * 2.0 ** -9: 2.0 ** -8,
             2.5 * 2.0 ** -9: 2.0 ** -8, 3.5 * 2.0 ** -9: 4 * 2.0 ** -9, 440.0: 448.0,
             424.0: 416.0, -12.5: -12.0, -13.5: -14.0, 450.0: 448.0}
    for x, want in cases.items():
        assert v[O.e4m3_round(np.array([x]))[0]] == want, x


def test_round_agrees_with_torch_float8():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 40, rng.standard_normal(5000) * 1e-2,
                        rng.uniform(-448, 448, 5000), [0.0, -0.0, 448.0, -448.0]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_round(x), ref)


def test_representable_values_round_trip():
    v = O.e4m3_values()
    codes = np.array([c for c in range(256) if not np.isnan(v[c])], dtype=np.uint8)
    assert np.array_equal(O.e4m3_round(v[codes]), codes)


def test_row_scale_and_error_bound():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((50, 3, 128)) * rng.uniform(0.01, 10, (50, 3, 1))).astype(np.float32)
    x[7, 1] = 0.0                                   # a zero row
    codes, s = O.fp8_encode_rows(x)
    amax = np.abs(x).max(axis=2)
    np.testing.assert_array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
    assert s[7, 1] == 0 and not codes[7, 1].any()
    y = O.fp8_decode_rows(codes, s)
    err = np.abs(y.astype(np.float64) - x)
    bound = 2.0 ** -4 * np.abs(x) + s[:, :, None] * 2.0 ** -10 + 1e-30
    assert np.all(err <= bound * (1 + 1e-6))
    # the row maximum maps to the largest code
    i = np.abs(x).reshape(-1, 128).argmax(axis=1)
    flat = codes.reshape(-1, 128)[np.arange(150), i] & 0x7F
    assert np.all(flat[np.abs(x).reshape(-1, 128).max(axis=1) > 0] == 0x7E)


def test_encode_rejects_out_of_range_rounding():
    with pytest.raises(ValueError):
        O.e4m3_round(np.array([464.0]))


def test_bf16_bits_agrees_with_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(10000) * 7, rng.standard_normal(1000) * 1e-30,
                        [0.0, -0.0, 1.0, -2.5, 65504.0]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits(x), ref)


def test_round_trip_is_idempotent():
    """Re-encoding a decoded page (bf16) gives the same codes and scales: the
    row maximum decodes back to itself (its code is 448 and 448 * s rounds to
    the bf16 maximum), so the scale repeats, and every decoded value is within
    a bf16 rounding (2^-9 relative) of an E4M3 value, far inside that value's
    rounding interval (2^-4 relative).  A page that leaves HBM twice in a
    compressed DRAM tier is therefore quantised once."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((200, 3, 128)) * np.exp(rng.standard_normal((200, 3, 1)) * 4.0)
    x[5, 1] = 0.0                                             # a zero row
    xb = O.bf16_bits(x.astype(np.float32))
    c1, s1 = O.fp8_encode_rows(xb)
    y = O.bf16_bits(O.fp8_decode_rows(c1, s1))
    c2, s2 = O.fp8_encode_rows(y)
    assert np.array_equal(s1, s2) and np.array_equal(c1, c2)
    assert np.array_equal(O.bf16_bits(O.fp8_decode_rows(c2, s2)), y)
