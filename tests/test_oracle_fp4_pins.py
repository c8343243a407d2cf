"""Pins for the oracle's NVFP4 page codec (the compressed DRAM tier's FP4 form:
E2M1 codes, E4M3 scales per 16-element block, one fp32 scale per row):
code values from the E2M1 field definitions, round-to-nearest-even checked
against a brute-force nearest search, scales computed by hand for constructed
rows, exact round trips of representable rows, an error bound that uses only
the input and the format (no intermediate of the codec), zero rows and the
nibble order.

CPU only; no GPU, no CUDA library."""

import numpy as np

import oracle as O

MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_from_format():
    v = O.e2m1_values()
    assert list(v[:8]) == MAGS                          # 0, subnormal 0.5, then 1 .. 6
    assert list(v[8:]) == [-m for m in MAGS] and np.signbit(v[8])
    assert v[0x2] == 1.0 and v[0x4] == 2.0 and v[0x7] == 6.0   # exponent bias 1


def _brute(q):
    """Nearest E2M1 magnitude by exhaustive search, ties to the even code,
    saturation at 6, sign kept."""
    out = []
    for x in np.asarray(q, dtype=np.float64).ravel():
        a = min(abs(x), 6.0)
        dist = [abs(a - m) for m in MAGS]
        best = min(range(8), key=lambda c: (dist[c], c % 2))
        neg = x < 0 or (x == 0 and np.signbit(x))
        out.append(best | (8 if neg else 0))
    return np.array(out, dtype=np.uint8)


def test_round_to_nearest_even():
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0,
             7.0: 6.0, 1e9: 6.0, 0.26: 0.5, 0.24: 0.0, 4.9: 4.0, 5.1: 6.0}
    v = O.e2m1_values()
    for q, want in cases.items():
        assert v[O.e2m1_round(np.array([q]))[0]] == want, q
        assert v[O.e2m1_round(np.array([-q]))[0]] == -want, -q
    grid = np.concatenate([np.linspace(-7, 7, 4001), np.array(MAGS), -np.array(MAGS), [-0.0]])
    assert np.array_equal(O.e2m1_round(grid), _brute(grid))


def test_scales_of_a_constructed_row():
    # two blocks of 16: block 0 holds the row maximum 2.625 = 2688 * 2^-10, block 1
    # reaches 2.625 / 4; g = 2^-10 exactly, block 0's scale 2.625 / (6 g) = 448,
    # block 1's 112 (both E4M3 values)
    row = np.zeros((1, 1, 32), dtype=np.float32)
    row[0, 0, 3] = -2.625
    row[0, 0, 16 + 5] = 2.625 / 4
    codes, sb, g = O.nvfp4_encode_rows(row)
    e4 = O.e4m3_values()
    assert g[0, 0] == np.float32(2.0 ** -10)
    assert e4[sb[0, 0, 0]] == 448.0 and e4[sb[0, 0, 1]] == 112.0
    # the maxima land on -6 and 6 (codes 0xF and 0x7); everything else is zero
    c = np.empty(32, dtype=np.uint8)
    c[0::2], c[1::2] = codes[0, 0] & 0xF, codes[0, 0] >> 4
    assert c[3] == 0xF and c[21] == 0x7 and (np.delete(c, [3, 21]) == 0).all()


def test_representable_rows_round_trip():
    # element scale 448 * 2^-10 = 0.4375 in both blocks: every E2M1 value times it
    # is an fp32 (and bf16) value, so the row decodes to itself
    rng = np.random.default_rng(5)
    es = 448.0 * 2.0 ** -10
    vals = O.e2m1_values()
    for _ in range(20):
        c = rng.integers(0, 16, size=(2, 3, 64))
        c[:, :, 0::16] = 7                               # each block reaches 6
        x = (vals[c] * es).astype(np.float32)
        codes, sb, g = O.nvfp4_encode_rows(x)
        y = O.nvfp4_decode_rows(codes, sb, g)
        assert np.array_equal(y, x)
        assert np.array_equal(O.bf16_bits(y), O.bf16_bits(x))


def test_error_bound():
    """|x - decode| <= max(es, |x|) / 4 with es <= (block max / 6) * 1.0625: the
    E2M1 half step is at most a quarter of the value (or of es below 1), the E4M3
    block scale is within 2^-4 of its target, and saturation past 6 stays
    inside the same bound."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((64, 4, 128)) * np.exp(rng.standard_normal((64, 4, 1)) * 3.0)
    x = x * np.exp(rng.standard_normal((64, 4, 128)) * 0.5)
    xb = O.decode_bf16(O.bf16_bits(x.astype(np.float32)))
    codes, sb, g = O.nvfp4_encode_rows(O.bf16_bits(x.astype(np.float32)))
    y = O.nvfp4_decode_rows(codes, sb, g).astype(np.float64)
    bmax = np.abs(xb).reshape(64, 4, 8, 16).max(axis=3)
    es_bound = np.repeat(bmax / 6.0 * 1.0625, 16, axis=2)
    bound = np.maximum(es_bound, np.abs(xb)) / 4.0 * (1 + 2.0 ** -18) + 1e-30
    assert (np.abs(y - xb) <= bound).all()
    # and the codec is not trivially exact: the bound is nearly reached somewhere
    assert (np.abs(y - xb) / bound).max() > 0.5


def test_zero_rows_and_nibble_order():
    x = np.zeros((2, 1, 16), dtype=np.float32)
    x[1, 0, :] = [6 * 2.0 ** -10 * v for v in (1, -1, 0.5, 2, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 3)]
    codes, sb, g = O.nvfp4_encode_rows(x)
    assert (codes[0] == 0).all() and (sb[0] == 0).all() and g[0, 0] == 0
    assert (O.nvfp4_decode_rows(codes, sb, g)[0] == 0).all()
    # element 0 in the low nibble of byte 0, element 1 in the high nibble
    vals = O.e2m1_values()
    dec = O.nvfp4_decode_rows(codes, sb, g)[1, 0]
    assert np.sign(dec[0]) == 1 and np.sign(dec[1]) == -1
    assert vals[codes[1, 0, 0] & 0xF] > 0 and vals[codes[1, 0, 0] >> 4] < 0
