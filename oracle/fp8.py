"""FP8 (e4m3) inputs for packed prefill -- TEST INFRASTRUCTURE (part of the oracle).

The page's abstract counts "selective FP8" among the engine's mixed-precision choices
without saying which matmuls use it.  The reading taken here for a future FP8 variant of the
packed prefill: Q and K arrive as 8-bit E4M3 codes with one power-of-two scale per tensor, V
stays bf16, and the attention is the same causal softmax attention over the dequantised
values.  (Only Q.K^T runs in FP8: quantising the softmax weights P to E4M3 for P.V as well
would put the output about 2e-2 RMS away from this result, beyond the parity bar.)

E4M3 (the OCP 8-bit floating-point format, "E4M3FN"): one sign bit, four exponent bits with
bias 7 and three mantissa bits.  Exponent field 0 holds the subnormals m/8 * 2^-6; the other
fields hold (1 + m/8) * 2^(e - 7).  There are no infinities; S.1111.111 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448.

Encoding rounds to the nearest representable value, ties to the even mantissa, and saturates
finite values beyond 448 to +-448 (the "satfinite" behaviour of the GPU's conversions).

A power-of-two scale keeps every dequantised value exactly representable in bf16 (3
mantissa bits fit in bf16's 7, and the exponent range of the scaled values stays inside
bf16's), so the fp64 prefill oracle of this package, which takes bf16 bit patterns, computes
the FP8 attention exactly from the dequantised inputs.  The pins are in
``tests/test_oracle_fp8_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F                 # positive NaN code; 0xFF is the negative one
_MIN_NORMAL_EXP = -6             # exponent of the smallest normal, 2^-6
_SUBNORMAL_STEP = 2.0 ** -9      # spacing of the subnormals, 2^-6 / 8


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each uint8 E4M3 code (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * _SUBNORMAL_STEP, np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64)))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def e4m3_encode(x) -> np.ndarray:
    """uint8 E4M3 code of each value: round to nearest, ties to even, finite values beyond
    448 saturate to +-448, NaN maps to the NaN code of its sign."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    # the spacing of representable values around a: 2^(e-3) for a in [2^e, 2^(e+1)), e >= -6;
    # 2^-9 below 2^-6 (subnormals)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, _MIN_NORMAL_EXP)
    step = np.ldexp(1.0, (e - 3).astype(np.int64))
    q = np.rint(a / step)                     # ties to even on the lattice of this binade
    # codes are contiguous in magnitude: a binade below 2^-6 holds codes 0..8, binade e holds
    # codes 8 * (e + 7) .. 8 * (e + 7) + 8 (the last one is the next binade's first)
    code = np.where(e == _MIN_NORMAL_EXP, q, 8.0 * (e + 7) + (q - 8.0))
    code = np.where(a == 0.0, 0.0, code).astype(np.int64)
    code = np.minimum(code, 0x7E)
    code = np.where(nan, E4M3_NAN, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def tensor_scale(x) -> float:
    """The smallest power of two s with max|x| / s <= 448 (1.0 for an all-zero tensor)."""
    amax = float(np.max(np.abs(np.asarray(x, dtype=np.float64)))) if np.size(x) else 0.0
    if amax == 0.0:
        return 1.0
    k = math.ceil(math.log2(amax / E4M3_MAX))
    s = math.ldexp(1.0, k)
    if amax / s > E4M3_MAX:                   # guard against rounding in log2
        s *= 2.0
    elif amax / (s / 2.0) <= E4M3_MAX:
        s /= 2.0
    return s


def quantize(x):
    """(codes, scale): per-tensor power-of-two scale, codes = E4M3 of x / scale."""
    s = tensor_scale(x)
    return e4m3_encode(np.asarray(x, dtype=np.float64) / s), s


def dequantize_bf16_bits(codes, scale: float) -> np.ndarray:
    """bf16 bit patterns (uint16) of decode(codes) * scale, exact for a power-of-two scale."""
    if scale <= 0.0 or math.frexp(scale)[0] != 0.5:
        raise ValueError("the scale must be a positive power of two")
    v = (e4m3_decode(codes) * scale).astype(np.float32)
    bits = v.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("a dequantised value is not representable in bf16")
    return (bits >> 16).astype(np.uint16)


def prefill_fp8(q_codes, q_scale, k_codes, k_scale, v, cu_seqlens, scale: float, want_lse: bool = False):
    """Packed causal GQA prefill with FP8 Q and K: the fp64 oracle on the exact dequantised
    Q and K (codes [T, H, d] uint8, one power-of-two scale per tensor) and the bf16 V (bit
    patterns, uint16 [T, Hkv, d])."""
    from . import prefill
    return prefill(dequantize_bf16_bits(q_codes, q_scale), dequantize_bf16_bits(k_codes, k_scale), v,
                   cu_seqlens, scale, want_lse=want_lse)
