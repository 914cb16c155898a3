"""bg_packed_prefill_attn_noalloc, the entry point for callers that cannot
allocate device memory (no workspace argument: its scratch is a fixed array
inside the library).  Its output must match the regular entry point's, within
the tolerance the other parity tests use, on two calls in a row -- the second
call reuses the array the first one left behind.  This file sorts last so a
run that stops at the first failure has already run every other test."""
import numpy as np
import pytest

from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


def _run(x, noalloc):
    import torch
    T, Hq, d = x["q"].shape
    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    cu = i32_dev(x["cu_seqlens"])
    out = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
    if noalloc:
        bg.bg_packed_prefill_attn_noalloc(q, k, v, cu, x["max_seqlen"], out, lse=lse)
    else:
        B = len(x["cu_seqlens"]) - 1
        ws = torch.empty(bg.bg_packed_prefill_workspace_size(B, T, x["max_seqlen"], Hq, x["Hkv"], d),
                         dtype=torch.uint8, device="cuda")
        bg.bg_packed_prefill_attn(q, k, v, cu, x["max_seqlen"], out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return from_dev(out), lse.cpu().numpy().astype(np.float64)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    build.build()
    bg.load()
    # first a larger problem, then a smaller one: the second call runs over
    # whatever the first left in the shared scratch array
    first = wl.make_prefill_inputs([700, 1, 129, 256, 0, 383, 64] * 3, 16, 8, 128, seeds=(91, 92, 93))
    second = wl.make_prefill_inputs([200, 17, 128], 16, 8, 128, seeds=(94, 95, 96))
    for i, x in enumerate((first, second)):
        ref, ref_lse = _run(x, noalloc=False)
        got, got_lse = _run(x, noalloc=True)
        assert_parity(got, ref, f"noalloc call {i + 1}")
        assert np.max(np.abs(got_lse - ref_lse)) <= 1e-3


def test_noalloc_rejects_problems_beyond_its_scratch():
    bg.load()
    fake = 0x10000
    # 200,000 sequences need more work-list entries than the fixed scratch holds
    st = bg.raw.bg_packed_prefill_attn_noalloc(fake, fake * 2, fake * 3, fake * 4, 200000, 200000, 1, 16, 8, 128,
                                               0.1, fake * 5, None, None, None)
    assert st == bg.BG_ERR_UNSUPPORTED
