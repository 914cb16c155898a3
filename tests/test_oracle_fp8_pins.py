"""Pins of the FP8 (E4M3) part of the oracle, each independent of its arithmetic:

* the values of codes named by the format (1.0, 2.0, the largest finite 448, the smallest
  normal 2^-6, the smallest subnormal 2^-9, NaN);
* every one of the 256 codes against torch's float8_e4m3fn (a library routine);
* encoding against a brute-force nearest-value search over the whole code table, ties to the
  even code, on random values and on every midpoint between neighbouring codes;
* saturation, signed zero and NaN;
* the per-tensor scale, the exactness of dequantisation in bf16 and the quantisation error
  bound (half a unit in the last place: 2^-4 relative for normal values);
* the prefill with FP8 Q and K against the independent padded-plus-mask formulation, and a
  length-1 sequence returning its own v row.
"""
import math

import numpy as np
import pytest

from oracle import fp8


def _bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_named_codes():
    d = fp8.e4m3_decode(np.array([0x38, 0x40, 0x7E, 0x08, 0x01, 0xB8, 0x00, 0x80, 0x07, 0x0F], dtype=np.uint8))
    assert d[0] == 1.0 and d[1] == 2.0 and d[2] == 448.0
    assert d[3] == 2.0 ** -6 and d[4] == 2.0 ** -9 and d[5] == -1.0
    assert d[6] == 0.0 and d[7] == 0.0 and math.copysign(1.0, d[7]) == -1.0
    assert d[8] == 7 * 2.0 ** -9                       # largest subnormal
    assert d[9] == 1.875 * 2.0 ** -6                   # exponent field 1, mantissa 7
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_every_code_against_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def test_encode_against_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(11)
    # torch maps values that round beyond 448 to NaN instead of saturating: stay below 464
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 100, 20000), rng.normal(0, 0.01, 20000),
                        rng.uniform(-463.9, 463.9, 20000)])
    x = x[np.abs(x) < 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), ref)


def _table():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def _nearest_brute(x, codes, vals):
    # nearest finite value; among equally near values the code with an even mantissa; a
    # signed zero keeps the sign of x
    out = []
    for xi in x:
        xi_c = min(max(xi, -fp8.E4M3_MAX), fp8.E4M3_MAX)
        dist = np.abs(vals - xi_c)
        best = np.flatnonzero(dist == dist.min())
        if len(best) > 1:
            best = [b for b in best if (int(codes[b]) & 1) == 0] or list(best)
        b = [c for c in best if bool(np.signbit(vals[c])) == bool(np.signbit(xi))] or list(best)
        out.append(int(codes[b[0]]))
    return np.array(out, dtype=np.uint8)


def test_encode_is_the_nearest_code_ties_to_even():
    codes, vals = _table()
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.normal(0, 4, 3000), rng.normal(0, 0.02, 1000), rng.uniform(-460, 460, 1000)])
    assert np.array_equal(fp8.e4m3_encode(x), _nearest_brute(x, codes, vals))


def test_every_midpoint_rounds_to_the_even_code():
    pos = np.arange(0x00, 0x7F, dtype=np.uint8)            # 0 .. 448, increasing
    v = fp8.e4m3_decode(pos)
    assert np.all(np.diff(v) > 0)
    mids = (v[:-1] + v[1:]) / 2
    got = fp8.e4m3_encode(mids).astype(np.int64)
    lo, hi = pos[:-1].astype(np.int64), pos[1:].astype(np.int64)
    want = np.where(lo % 2 == 0, lo, hi)
    assert np.array_equal(got, want)
    assert np.array_equal(fp8.e4m3_encode(-mids).astype(np.int64), want | 0x80)
    # every representable value encodes to itself
    assert np.array_equal(fp8.e4m3_encode(v), pos)


def test_saturation_zero_and_nan():
    got = fp8.e4m3_encode(np.array([449.0, 463.9, 464.0, 1e6, np.inf, -1e6, -np.inf, 0.0, -0.0, np.nan, -np.nan]))
    assert got.tolist()[:7] == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[7] == 0x00 and got[8] == 0x80
    assert (got[9] & 0x7F) == 0x7F and (got[10] & 0x7F) == 0x7F


def test_tensor_scale_is_the_smallest_fitting_power_of_two():
    rng = np.random.default_rng(13)
    for sigma in (1e-4, 0.3, 1.0, 7.0, 448.0, 1e5):
        x = rng.normal(0, sigma, 4096)
        s = fp8.tensor_scale(x)
        assert math.frexp(s)[0] == 0.5
        amax = np.abs(x).max()
        assert amax / s <= 448.0 < amax / (s / 2)
    assert fp8.tensor_scale(np.zeros(8)) == 1.0
    assert fp8.tensor_scale(np.array([448.0])) == 1.0 and fp8.tensor_scale(np.array([448.5])) == 2.0


def test_dequantisation_is_exact_in_bf16_and_within_half_an_ulp():
    rng = np.random.default_rng(14)
    x = rng.normal(0, 1.7, (64, 8, 32))
    codes, s = fp8.quantize(x)
    bits = fp8.dequantize_bf16_bits(codes, s)
    xh = _bf16_bits_to_f64(bits)
    assert np.array_equal(xh, fp8.e4m3_decode(codes) * s)
    y = np.abs(x) / s
    normal = y >= 2.0 ** -6
    err = np.abs(xh - x)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-12))
    assert np.all(err[~normal] <= s * 2.0 ** -10 * (1 + 1e-12))
    with pytest.raises(ValueError):
        fp8.dequantize_bf16_bits(codes, 0.3)


def test_fp8_prefill_against_the_padded_formulation():
    from oracle import oracle_np
    rng = np.random.default_rng(15)
    lengths = [1, 5, 17, 40]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 16
    # inputs that are exactly representable: random codes (no NaN) and power-of-two scales
    def codes(shape):
        c = rng.integers(0, 0x7F, size=shape).astype(np.uint8) | (rng.integers(0, 2, size=shape) * 0x80).astype(np.uint8)
        return c
    qc, kc = codes((T, Hq, d)), codes((T, Hkv, d))
    vb = (rng.normal(0, 1, (T, Hkv, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # bf16 V
    sq, sk = 2.0 ** -6, 2.0 ** -7
    got = fp8.prefill_fp8(qc, sq, kc, sk, vb, cu, 1 / math.sqrt(d))
    # the independent padded-plus-mask numpy formulation on the same dequantised values
    ref = oracle_np.prefill_padded(fp8.dequantize_bf16_bits(qc, sq), fp8.dequantize_bf16_bits(kc, sk), vb, cu,
                                   1 / math.sqrt(d))
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    # a length-1 sequence returns its own v row
    v0 = _bf16_bits_to_f64(vb[0])
    assert np.array_equal(got[0], np.repeat(v0, Hq // Hkv, axis=0))
