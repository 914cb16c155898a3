"""GPU parity of bg_packed_prefill_attn_fp8 (through the C ABI) against the fp64 oracle.

The reading (the abstract of "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化" names
"selective FP8" without saying which matmuls use it): Q and K arrive as E4M3 codes with one
power-of-two scale per tensor, V stays bf16, and the result is the causal attention over the
dequantised values, which oracle.fp8.prefill_fp8 computes exactly in fp64.  The codes are the
oracle's own quantisation (oracle.fp8: the tensor's power-of-two scale, then E4M3 round to
nearest even) of the usual seeded bf16 N(0,1) inputs; both sides get the same codes.  The bar
is the one every other parity test uses: max_abs <= 2e-2 and rel_rms <= 5e-3 per call."""
import math

import numpy as np
import pytest

import oracle
import oracle.fp8 as ofp8
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def quantize_bits(bits, chunk=1 << 26):
    """The oracle's per-tensor quantisation of bf16 bit patterns: scale = the smallest power
    of two with max|x| / scale <= 448, codes = E4M3(x / scale).  x / scale is exact for a
    power-of-two scale, so E4M3(x / scale) is a function of the bf16 pattern alone: the codes
    come from a 65,536-entry table of the oracle's encoder, applied in chunks."""
    flat = bits.reshape(-1)
    mag = 0
    for i in range(0, flat.size, chunk):
        mag = max(mag, int(np.max(flat[i:i + chunk] & 0x7FFF)))
    amax = float(np.array([mag << 16], dtype=np.uint32).view(np.float32)[0])
    scale = ofp8.tensor_scale(np.array([amax]))
    all_bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):                 # the NaN patterns map to the NaN code
        vals = (all_bits << 16).view(np.float32).astype(np.float64)
    table = ofp8.e4m3_encode(vals / scale)
    codes = np.empty(flat.size, dtype=np.uint8)
    for i in range(0, flat.size, chunk):
        codes[i:i + chunk] = table[flat[i:i + chunk]]
    return codes.reshape(bits.shape), scale


def fp8_inputs(x):
    qc, qs = quantize_bits(x["q"])
    kc, ks = quantize_bits(x["k"])
    return qc, qs, kc, ks


def u8_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def run_fp8(x, codes, want_lse=False):
    import torch
    qc, qs, kc, ks = codes
    T, Hq, d = x["q"].shape
    B = len(x["cu_seqlens"]) - 1
    out_full = torch.full((T * Hq * d + GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    out = out_full[:T * Hq * d].view(torch.bfloat16).view(T, Hq, d)
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(B, T, x["max_seqlen"], Hq, x["Hkv"], d),
                     dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_attn_fp8(u8_dev(qc), qs, u8_dev(kc), ks, to_dev(x["v"]), i32_dev(x["cu_seqlens"]),
                                  x["max_seqlen"], out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert np.all(out_full[T * Hq * d:].cpu().numpy() == SENTINEL), "write past the end of out"
    return out, lse


def check(x, what, want_lse=False, rows=None):
    codes = fp8_inputs(x)
    qc, qs, kc, ks = codes
    scale = 1.0 / math.sqrt(x["head_dim"])
    out, lse = run_fp8(x, codes, want_lse=want_lse)
    got = from_dev(out)
    if rows is None:
        if want_lse:
            ref, ref_lse = ofp8.prefill_fp8(qc, qs, kc, ks, x["v"], x["cu_seqlens"], scale, want_lse=True)
            lse_got = lse.cpu().numpy().astype(np.float64)
            assert np.max(np.abs(lse_got - ref_lse)) < 1e-3 * max(1.0, np.max(np.abs(ref_lse)))
        else:
            ref = ofp8.prefill_fp8(qc, qs, kc, ks, x["v"], x["cu_seqlens"], scale)
        return assert_parity(got, ref, what)
    idx, sub_cu = rows
    ref = ofp8.prefill_fp8(qc[idx], qs, kc[idx], ks, x["v"][idx], sub_cu, scale)
    assert np.all(np.isfinite(got))
    return assert_parity(got[idx], ref, what)


def test_fp8_tiny_config_parity():
    x = wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["tiny"])
    check(x, "fp8 tiny {17,64,100,211}", want_lse=True)


@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (8, 8), (6, 2), (16, 1)])
def test_fp8_ragged_tiles_parity(Hq, Hkv):
    lengths = [1, 2, 127, 128, 129, 255, 256, 257, 300, 0, 5, 384, 0, 77]
    x = wl.make_prefill_inputs(lengths, Hq, Hkv, 128, seeds=(111, 112, 113))
    check(x, f"fp8 ragged Hq{Hq} Hkv{Hkv}")


def test_fp8_long_and_outlier_parity():
    x = wl.make_prefill_inputs([2048, 1000, 1, 640], 16, 8, 128, seeds=(121, 122, 123))
    check(x, "fp8 long")
    y = wl.make_prefill_inputs([513, 700, 33], 16, 8, 128, seeds=(131, 132, 133), outlier_frac=0.05,
                               outlier_scale=8.0)
    check(y, "fp8 outliers", want_lse=True)


def test_fp8_length_one_returns_its_value_row():
    """One key: the softmax weight is exactly 1, so every output row is its own bf16 v row."""
    x = wl.make_prefill_inputs([1] * 21, 16, 8, 128, seeds=(141, 142, 143))
    out, _ = run_fp8(x, fp8_inputs(x))
    b = bits_from_dev(out)
    for t in range(21):
        for h in range(16):
            np.testing.assert_array_equal(b[t, h], x["v"][t, h // 2])


def test_fp8_matches_bf16_kernel_on_dequantised_inputs():
    """The same attention through the bf16 kernel on the exactly dequantised Q and K: the two
    kernels differ only in the operand format of Q.K^T, so they agree closely."""
    import torch
    x = wl.make_prefill_inputs([300, 17, 128, 129, 500], 16, 8, 128, seeds=(151, 152, 153))
    codes = fp8_inputs(x)
    qc, qs, kc, ks = codes
    out8, _ = run_fp8(x, codes)
    T, Hq, d = x["q"].shape
    out16 = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(5, T, 500, Hq, 8, d), dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_attn(to_dev(ofp8.dequantize_bf16_bits(qc, qs)), to_dev(ofp8.dequantize_bf16_bits(kc, ks)),
                              to_dev(x["v"]), i32_dev(x["cu_seqlens"]), 500, out16, workspace=ws)
    torch.cuda.synchronize()
    a, b = from_dev(out8), from_dev(out16)
    assert np.max(np.abs(a - b)) <= 1e-2
    assert np.sqrt(np.sum((a - b) ** 2) / np.sum(b * b)) <= 2e-3


def test_fp8_prefill_only_config_full_parity():
    x = wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["prefill_only"], layer=0)
    check(x, "fp8 prefill_only full")


def test_fp8_skewed_config_sampled_parity():
    """The full skewed stress layer launched as the benchmark launches it; the oracle recomputes
    the longest, the shortest and a seeded random set of sequences."""
    cfg = wl.PREFILL_CONFIGS["skewed"]
    x = wl.make_prefill_config_inputs(cfg)
    L = np.array(x["lengths"])
    cu = x["cu_seqlens"]
    order = np.argsort(L)
    rng = np.random.default_rng(78)
    pick = sorted(set(order[-3:].tolist() + order[:3].tolist() + rng.choice(len(L), 24, replace=False).tolist()))
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in pick])
    sub_cu = wl.cu_from_lengths([int(L[i]) for i in pick])
    check(x, "fp8 skewed sampled", rows=(idx, sub_cu))
