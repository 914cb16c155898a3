"""GPU parity of bg_packed_last_token_attn (through the C ABI): the attention
output of each packed sequence's last valid token, against the fp64 oracle on
the same seeded bf16 inputs, and against the last rows of the GPU prefill."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0x7FC1                 # a bf16 NaN pattern the kernel never writes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def last_rows(x):
    """q of each sequence's last valid token (row 0 stands in for empty sequences)."""
    cu = x["cu_seqlens"]
    idx = [max(int(cu[i + 1]) - 1, 0) for i in range(len(cu) - 1)]
    return np.ascontiguousarray(x["q"][idx])


def run_last(x, want_lse=False, dev_status=None, cu_override=None):
    import torch
    B = len(x["cu_seqlens"]) - 1
    Hq, d = x["Hq"], x["head_dim"]
    q = to_dev(last_rows(x))
    k, v = to_dev(x["k"]), to_dev(x["v"])
    cu = i32_dev(x["cu_seqlens"] if cu_override is None else cu_override)
    n = B * Hq * d
    full = torch.full((n + GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    out = full[:n].view(torch.bfloat16).view(B, Hq, d)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    bg.bg_packed_last_token_attn(q, k, v, cu, x["max_seqlen"], out, lse=lse, dev_status=dev_status)
    torch.cuda.synchronize()
    assert np.all(full[n:].cpu().numpy() == SENTINEL), "write past the end of out"
    return out, lse


def check(x, what, want_lse=False):
    scale = 1.0 / math.sqrt(x["head_dim"])
    out, lse = run_last(x, want_lse=want_lse)
    ref, ref_lse = oracle.last_token(last_rows(x), x["k"], x["v"], x["cu_seqlens"], scale, want_lse=True)
    lengths = np.diff(x["cu_seqlens"])
    got = from_dev(out)
    live = lengths > 0
    assert np.all(bits_from_dev(out)[~live] == SENTINEL), f"{what}: an empty sequence's row was written"
    assert_parity(got[live], ref[live], what)
    if want_lse:
        lg = lse.cpu().numpy().astype(np.float64)[live]
        assert np.max(np.abs(lg - ref_lse[live])) < 1e-3 * max(1.0, np.max(np.abs(ref_lse[live])))


def test_last_token_tiny_with_lse():
    check(wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["tiny"]), "tiny", want_lse=True)


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 8, 128), (14, 2, 64), (16, 1, 128), (4, 4, 64), (48, 3, 128)])
def test_last_token_ragged_chunks(Hq, Hkv, d):
    """Lengths around the 256-key chunk and far beyond it, with empty sequences."""
    lengths = [0, 1, 2, 255, 256, 257, 0, 511, 513, 1000, 2048, 3]
    x = wl.make_prefill_inputs(lengths, Hq, Hkv, d, seeds=(91, 92, 93))
    check(x, f"ragged Hq{Hq} Hkv{Hkv} d{d}", want_lse=True)


def test_last_token_prefill_only_config():
    check(wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["prefill_only"]), "prefill_only")


def test_last_token_skewed_config_full():
    check(wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["skewed"]), "skewed")


def test_last_token_equals_last_rows_of_gpu_prefill():
    """The same rows of bg_packed_prefill_attn: both kernels against each other."""
    import torch
    x = wl.make_prefill_inputs([37, 128, 300, 1, 700], 16, 8, 128, seeds=(95, 96, 97))
    T = x["q"].shape[0]
    out_full = torch.empty((T, 16, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(5, T, x["max_seqlen"], 16, 8, 128), dtype=torch.uint8,
                     device="cuda")
    cu = i32_dev(x["cu_seqlens"])
    bg.bg_packed_prefill_attn(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), cu, x["max_seqlen"], out_full,
                              workspace=ws)
    out_last, _ = run_last(x)
    rows = [int(c) - 1 for c in x["cu_seqlens"][1:]]
    pre = from_dev(out_full)[rows]
    assert_parity(from_dev(out_last), pre, "last token vs prefill last rows")


def test_last_token_bad_cu_seqlens_reported():
    import torch
    x = wl.make_prefill_inputs([10, 20, 30], 16, 8, 128, seeds=(1, 2, 3))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = np.array([0, 25, 20, 60], np.int32)      # not monotone in the middle
    out, _ = run_last(x, dev_status=st, cu_override=bad)
    assert int(st.item()) & bg.BG_DEVSTAT_CU_SEQLENS
    assert np.all(bits_from_dev(out)[1] == SENTINEL)   # the bad sequence wrote nothing
