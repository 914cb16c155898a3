"""Failure path on the GPU without a fault: a bounded pipeline wait that runs out.

bg_selftest_wait_timeout waits, through the same bounded-wait routine every pipeline wait of
the attention kernels uses, on an mbarrier that nothing arrives on.  The wait must end after
the library's limit (about one second), report BG_DEVSTAT_TIMEOUT to the host, and leave the
context usable: a prefill call right after it still matches the oracle."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def test_bounded_wait_runs_out_and_context_survives():
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    bg.bg_selftest_wait_timeout(st, waited)
    torch.cuda.synchronize()
    assert int(st.item()) == bg.BG_DEVSTAT_TIMEOUT
    ns = int(waited.item())
    assert 0.9e9 <= ns <= 3e9, ns          # the limit is one second of device time
    # the same context runs the hot path correctly afterwards
    x = wl.make_prefill_config_inputs(wl.PREFILL_CONFIGS["tiny"])
    T, Hq, d = x["q"].shape
    out = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(len(x["cu_seqlens"]) - 1, T, x["max_seqlen"], Hq, x["Hkv"], d),
                     dtype=torch.uint8, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bg_packed_prefill_attn(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), i32_dev(x["cu_seqlens"]),
                              x["max_seqlen"], out, workspace=ws, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], 1 / math.sqrt(d))
    assert_parity(from_dev(out), ref, "prefill after a timed-out wait")
