"""Pins for the oracle's e4m3 storage format and its use in attention (CPU only)."""
import numpy as np
import pytest

from oracle import attention as oatt
from oracle import fp8


def test_decode_table_spot_values():
    v = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9        # subnormals
    assert v[0x08] == 2.0 ** -6                                      # smallest normal
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0x3F] == 1.875
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0                    # largest finite
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])                   # the only NaN codes
    assert np.sum(np.isnan(v)) == 2 and np.all(np.isfinite(v[~np.isnan(v)]))


def test_positive_codes_are_ordered_by_value():
    v = fp8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)


def test_every_finite_code_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    v = fp8.e4m3_decode(codes)
    fin = ~np.isnan(v)
    assert np.array_equal(fp8.e4m3_encode(v[fin].astype(np.float32)), codes[fin])


def test_rounding_is_to_nearest_with_ties_to_even():
    enc = lambda x: int(fp8.e4m3_encode(np.float32([x]))[0])
    assert enc(1.0625) == 0x38          # halfway 1.0 / 1.125: even mantissa (1.0)
    assert enc(1.1875) == 0x3A          # halfway 1.125 / 1.25: even mantissa (1.25)
    assert enc(1.0626) == 0x39          # just above halfway
    assert enc(2.0 ** -10) == 0x00      # halfway 0 / 2^-9: even (0)
    assert enc(3 * 2.0 ** -10) == 0x02  # halfway 2^-9 / 2^-8: even (2^-8)
    assert enc(-1.0625) == 0xB8


def test_saturation_and_nan():
    enc = lambda x: int(fp8.e4m3_encode(np.float32([x]))[0])
    assert enc(448.0) == 0x7E and enc(460.0) == 0x7E and enc(1e30) == 0x7E
    assert enc(-1e30) == 0xFE and enc(np.inf) == 0x7E and enc(-np.inf) == 0xFE
    assert enc(np.nan) == 0x7F


def test_encoder_agrees_with_torch_inside_the_finite_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(200000) * s for s in (0.01, 1.0, 60.0)]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]           # torch's float8_e4m3fn does not saturate beyond
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def test_quantize_divides_in_float32_then_rounds():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(5000).astype(np.float32)
    scale = np.float32(0.0137)
    assert np.array_equal(fp8.quantize(x, scale), fp8.e4m3_encode(x / scale))
    codes = fp8.quantize(x, scale)
    back = fp8.dequantize(codes, scale)
    # half a step of 3 mantissa bits, relative, except near zero
    big = np.abs(x) > 2.0 ** -6 * scale
    assert np.all(np.abs(back[big] - x[big]) <= np.abs(x[big]) * 2.0 ** -4 + 1e-12)


def test_paged_attention_over_fp8_values_equals_contiguous():
    rng = np.random.default_rng(10)
    B, hkv, D, nb = 4, 2, 8, 12
    kc = rng.integers(0, 256, size=(nb, hkv, B, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(nb, hkv, B, D), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x01      # no NaN codes
    vc[(vc & 0x7F) == 0x7F] = 0x01
    k = fp8.dequantize(kc, 0.01)
    v = fp8.dequantize(vc, 0.02)
    tables = np.array([[3, 7, 1], [0, 5, -1]], dtype=np.int32)
    lens = np.array([10, 6], dtype=np.int32)
    q = rng.standard_normal((2, 4, D))
    out = oatt.paged_decode(q, k, v, tables, lens, 0.3, hkv)
    kseq = [np.concatenate([k[b] .transpose(1, 0, 2) for b in t[t >= 0]])[:L] for t, L in zip(tables, lens)]
    vseq = [np.concatenate([v[b] .transpose(1, 0, 2) for b in t[t >= 0]])[:L] for t, L in zip(tables, lens)]
    ref = oatt.contiguous_decode(q, kseq, vseq, 0.3, hkv)
    assert np.array_equal(out, ref)


def test_encoder_is_the_brute_force_nearest_value():
    """For values across every binade (and exact midpoints), the code is the
    finite e4m3 value nearest to y, the even code on a tie, +-448 beyond 448:
    checked against a search over all 254 finite codes."""
    rng = np.random.default_rng(11)
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    fc, fv = codes[fin], vals[fin]
    mags = np.exp2(rng.uniform(-12, 9.5, 20000))
    pos = np.sort(np.unique(np.abs(fv)))
    mids = (pos[:-1] + pos[1:]) / 2                         # exact in float32
    y = np.concatenate([mags, -mags, mids, -mids]).astype(np.float32)
    got = fp8.e4m3_encode(y)
    yy = np.minimum(np.abs(y.astype(np.float64)), 448.0) * np.where(np.signbit(y), -1.0, 1.0)
    d = np.abs(yy[:, None] - fv[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equally near codes take the even one (the sign of zero follows y)
    even = cand & ((fc[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1, keepdims=True), even, cand)
    sign_ok = (fc[None, :] >> 7) == np.signbit(y)[:, None]
    pick = pick & np.where((fv[None, :] == 0), sign_ok, True)
    want = fc[np.argmax(pick, axis=1)]
    assert np.array_equal(got, want)
