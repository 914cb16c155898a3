"""bg_packed_prefill_attn_noalloc, the entry point for callers that cannot
allocate device memory (no workspace argument: its scratch is a fixed array
inside the library).  It runs the same kernels as the regular entry point, so
on two calls in a row -- the second reusing the array the first one left
behind -- its output and LSE must be bit-identical to the regular entry
point's; one of the calls is also compared with the fp64 oracle at the
parity tolerance.  Its host-side rejections are tested without a GPU in
tests/test_abi_host.py.  This file sorts last so a run that stops at the
first failure has already run every other test."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

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
    return bits_from_dev(out), lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    build.build()
    bg.load()
    # first a larger problem, then a smaller one: the second call runs over
    # whatever the first left in the shared scratch array
    first = wl.make_prefill_inputs([700, 1, 129, 256, 0, 383, 64] * 3, 16, 8, 128, seeds=(91, 92, 93))
    second = wl.make_prefill_inputs([200, 17, 128], 16, 8, 128, seeds=(94, 95, 96))
    for i, x in enumerate((first, second)):
        ref_bits, ref_lse = _run(x, noalloc=False)
        got_bits, got_lse = _run(x, noalloc=True)
        assert np.array_equal(got_bits, ref_bits), f"noalloc call {i + 1}: output differs from the workspace call"
        assert np.array_equal(got_lse.view(np.uint32), ref_lse.view(np.uint32)), f"noalloc call {i + 1}: lse differs"
        if i == 1:
            want = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], 1.0 / math.sqrt(128))
            got = (got_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            assert_parity(got, want, "noalloc call 2 vs oracle")
