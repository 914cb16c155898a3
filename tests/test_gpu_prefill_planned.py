"""GPU check of the two-part prefill (bg_packed_prefill_plan once, then
bg_packed_prefill_attn_planned per layer) through the C ABI.

One packing serves every layer of a batch, so its work list is built once.  Checked:
  * each planned run is bit-identical to the one-call bg_packed_prefill_attn on the same
    layer, over several layers that share one plan (and lse too);
  * a planned layer matches the fp64 oracle within the parity tolerance;
  * a plan whose cu_seqlens fail the device checks flags dev_status, and the planned run
    after it writes nothing, as the one-call form does;
  * a planned run given another packing's plan (other total tokens and sequence count)
    writes nothing and raises BG_DEVSTAT_PLAN."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def _layer_inputs(lengths, Hq, Hkv, d, layer):
    return wl.make_prefill_inputs(lengths, Hq, Hkv, d, seeds=(401 + 3 * layer, 402 + 3 * layer, 403 + 3 * layer))


@pytest.mark.parametrize("Hq,Hkv,d", [(16, 8, 128), (12, 4, 64)])
def test_planned_runs_match_the_one_call_form(Hq, Hkv, d):
    import torch
    lengths = [300, 1, 0, 129, 64, 511, 17, 256]
    xs = [_layer_inputs(lengths, Hq, Hkv, d, layer) for layer in range(3)]
    cu_np = xs[0]["cu_seqlens"]
    T, B, maxlen = int(cu_np[-1]), len(lengths), max(lengths)
    cu = i32_dev(cu_np)
    ws_plan = torch.empty(bg.bg_packed_prefill_workspace_size(B, T, maxlen, Hq, Hkv, d), dtype=torch.uint8,
                          device="cuda")
    ws_one = torch.empty_like(ws_plan)
    bg.bg_packed_prefill_plan(cu, T, maxlen, workspace=ws_plan)
    outs = []
    for x in xs:
        q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
        a = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        b = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        la = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
        lb = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
        bg.bg_packed_prefill_attn_planned(q, k, v, cu, maxlen, a, lse=la, workspace=ws_plan)
        bg.bg_packed_prefill_attn(q, k, v, cu, maxlen, b, lse=lb, workspace=ws_one)
        torch.cuda.synchronize()
        assert np.array_equal(bits_from_dev(a), bits_from_dev(b)), "planned output differs from the one-call form"
        assert torch.equal(la, lb), "planned lse differs from the one-call form"
        outs.append(a)
    x = xs[2]
    ref = oracle.prefill(x["q"], x["k"], x["v"], cu_np, 1.0 / math.sqrt(d))
    assert_parity(from_dev(outs[2]), ref, f"planned layer 2 Hq{Hq} Hkv{Hkv} d{d}")


def test_a_bad_plan_makes_the_planned_run_write_nothing():
    import torch
    lengths = [40, 70]
    x = _layer_inputs(lengths, 16, 8, 128, 0)
    T = int(x["cu_seqlens"][-1])
    bad = np.array([0, 80, 70], dtype=np.int32)           # decreasing: the device check fails
    cu = i32_dev(bad)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(2, T, 80, 16, 8, 128), dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_plan(cu, T, 80, workspace=ws, dev_status=st)
    out = torch.full((T, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    bg.bg_packed_prefill_attn_planned(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), cu, 80, out, workspace=ws,
                                      dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bg.BG_DEVSTAT_CU_SEQLENS
    assert torch.isnan(out.float()).all(), "a planned run after a failed plan wrote output"


def test_a_plan_for_another_packing_is_refused():
    # plan 2 sequences (300 tokens), then run on 3 sequences (500 tokens): the run writes nothing
    # and raises BG_DEVSTAT_PLAN.  (The planned list only addresses rows below 300, inside the
    # larger run's buffers, so even an unchecked run would stay in bounds.)
    import torch
    a = _layer_inputs([100, 200], 16, 8, 128, 0)
    b = _layer_inputs([100, 200, 200], 16, 8, 128, 1)
    Ta, Tb = int(a["cu_seqlens"][-1]), int(b["cu_seqlens"][-1])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(3, Tb, 200, 16, 8, 128), dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_plan(i32_dev(a["cu_seqlens"]), Ta, 200, workspace=ws, dev_status=st)
    out = torch.full((Tb, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    bg.bg_packed_prefill_attn_planned(to_dev(b["q"]), to_dev(b["k"]), to_dev(b["v"]), i32_dev(b["cu_seqlens"]), 200,
                                      out, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == bg.BG_DEVSTAT_PLAN
    assert torch.isnan(out.float()).all(), "a run with another packing's plan wrote output"
