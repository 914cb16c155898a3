"""GPU parity of bg_packed_prefill_attn (through the C ABI) against the fp64
oracle on the same seeded bf16 inputs.  Tolerances: max_abs <= 2e-2 and
rel_rms <= 5e-3 over each call's output."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096                      # canary elements after every output buffer
SENTINEL = 0x7FC1                 # a bf16 NaN pattern the kernels never write


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def run_prefill(x, scale=None, want_lse=False, dev_status=None, cu_override=None):
    import torch
    T, Hq, d = x["q"].shape
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    cu = i32_dev(x["cu_seqlens"] if cu_override is None else cu_override)
    B = len(x["cu_seqlens"]) - 1
    out_full = torch.full((T * Hq * d + GUARD,), 0, dtype=torch.int16, device="cuda")
    out_full.fill_(SENTINEL - 65536 if SENTINEL > 32767 else SENTINEL)
    out = out_full[:T * Hq * d].view(torch.bfloat16).view(T, Hq, d)
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(B, T, x["max_seqlen"], Hq, x["Hkv"], d),
                     dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_attn(q, k, v, cu, x["max_seqlen"], out, lse=lse, scale=scale, workspace=ws,
                              dev_status=dev_status)
    torch.cuda.synchronize()
    guard = out_full[T * Hq * d:].cpu().numpy()
    assert np.all(guard == SENTINEL), "write past the end of out"
    return out, lse


def check_against_oracle(x, what, want_lse=False):
    d = x["head_dim"]
    scale = 1.0 / math.sqrt(d)
    out, lse = run_prefill(x, want_lse=want_lse)
    got = from_dev(out)
    if want_lse:
        ref, ref_lse = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale, want_lse=True)
        lse_got = lse.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(lse_got - ref_lse)) < 1e-3 * max(1.0, np.max(np.abs(ref_lse)))
    else:
        ref = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    return assert_parity(got, ref, what)


def test_tiny_config_parity():
    x = wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["tiny"])
    check_against_oracle(x, "tiny {17,64,100,211}", want_lse=True)


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 8, 128), (16, 8, 64), (8, 8, 128), (12, 4, 64), (6, 2, 128), (16, 1, 64)])
def test_ragged_tiles_parity(Hq, Hkv, d):
    lengths = [1, 2, 127, 128, 129, 255, 256, 257, 300, 0, 5, 384, 0, 77]
    x = wl.make_prefill_inputs(lengths, Hq, Hkv, d, seeds=(11, 12, 13))
    check_against_oracle(x, f"ragged Hq{Hq} Hkv{Hkv} d{d}")


def test_long_sequences_parity():
    lengths = [2048, 1000, 1, 640]
    x = wl.make_prefill_inputs(lengths, 16, 8, 128, seeds=(21, 22, 23))
    check_against_oracle(x, "long")


@pytest.mark.parametrize("seeds,scale_k", [((31, 32, 33), 8.0), ((131, 132, 133), 8.0), ((231, 232, 233), 8.0),
                                           ((331, 332, 333), 16.0)])
def test_outlier_logits_parity(seeds, scale_k):
    """Peaked softmax rows (5 % of K rows scaled up): the dominant weight's bf16 rounding must
    not move the row (the normaliser sums the same rounded weights that P.V uses)."""
    lengths = [513, 700, 33]
    x = wl.make_prefill_inputs(lengths, 16, 8, 128, seeds=seeds, outlier_frac=0.05, outlier_scale=scale_k)
    check_against_oracle(x, f"outliers {seeds} x{scale_k}", want_lse=True)


def test_length_one_is_exact_and_deterministic():
    x = wl.make_prefill_inputs([1] * 37 + [3], 16, 8, 128, seeds=(41, 42, 43))
    out1, _ = run_prefill(x)
    out2, _ = run_prefill(x)
    b1, b2 = bits_from_dev(out1), bits_from_dev(out2)
    np.testing.assert_array_equal(b1, b2)
    # a single key: the output is that key's value row, bit for bit
    for t in range(37):
        for h in range(16):
            np.testing.assert_array_equal(b1[t, h], x["v"][t, h // 2])


def test_causality_bitexact_on_gpu():
    x = wl.make_prefill_inputs([300], 4, 2, 128, seeds=(51, 52, 53))
    base = bits_from_dev(run_prefill(x)[0])
    p = 140
    y = dict(x)
    y["k"] = x["k"].copy()
    y["v"] = x["v"].copy()
    y["k"][p + 1:] = x["k"][::-1][: 300 - p - 1]
    y["v"][p + 1:] = x["v"][::-1][: 300 - p - 1]
    pert = bits_from_dev(run_prefill(y)[0])
    np.testing.assert_array_equal(pert[:p + 1], base[:p + 1])
    assert np.any(pert[p + 1:] != base[p + 1:])


def test_bad_cu_seqlens_reported_and_nothing_written():
    import torch
    x = wl.make_prefill_inputs([100, 50, 20], 4, 2, 64, seeds=(61, 62, 63))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = np.array([0, 100, 90, 170], np.int32)                   # decreasing
    out, _ = run_prefill(x, dev_status=st, cu_override=bad)
    assert int(st.item()) & bg.BG_DEVSTAT_CU_SEQLENS
    assert np.all(bits_from_dev(out) == SENTINEL)
    st.zero_()
    x2 = dict(x)
    x2["max_seqlen"] = 60                                          # 100 > max_seqlen
    out2, _ = run_prefill(x2, dev_status=st)
    assert int(st.item()) & bg.BG_DEVSTAT_SEQ_TOO_LONG
    assert np.all(bits_from_dev(out2) == SENTINEL)


def test_prefill_only_config_full_parity():
    """Full-size Prefill-Only batch (240 sequences, T = 70,375), one layer,
    every output row compared with the oracle."""
    x = wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["prefill_only"], layer=0)
    check_against_oracle(x, "prefill_only full")


def test_skewed_config_sampled_parity():
    """Full-size skewed stress (4096 sequences, T = 1,356,586) launched as the
    benchmark launches it; the oracle recomputes a sample of sequences (the
    longest, the shortest and a seeded random set), whose rows are compared."""
    cfg = wl.PREFILL_CONFIGS["skewed"]
    x = wl.make_prefill_config_inputs(cfg)
    out, _ = run_prefill(x)
    got = from_dev(out)
    L = np.array(x["lengths"])
    cu = x["cu_seqlens"]
    order = np.argsort(L)
    rng = np.random.default_rng(77)
    pick = sorted(set(order[-3:].tolist() + order[:3].tolist() + rng.choice(len(L), 24, replace=False).tolist()))
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in pick])
    sub_cu = wl.cu_from_lengths([int(L[i]) for i in pick])
    ref = oracle.prefill(x["q"][idx], x["k"][idx], x["v"][idx], sub_cu, 1.0 / math.sqrt(cfg.head_dim))
    assert_parity(got[idx], ref, "skewed sampled")
    assert np.all(np.isfinite(got))
