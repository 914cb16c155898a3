"""GPU parity of the beam-search decode path through the C ABI:
bg_beam_suffix_reorder (bit-exact against the oracle's explicit per-beam
histories) and bg_beam_decode_attn (against the fp64 oracle over
[shared prompt ; the beam's own suffix])."""
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


class GpuBeams:
    """Device-side state of one decode: ping-pong suffix buffers."""

    def __init__(self, pr, suffix_max):
        import torch
        R, W, Hkv, d = pr["R"], pr["W"], pr["Hkv"], pr["head_dim"]
        self.pr = pr
        self.S = suffix_max
        shape = (R, W, suffix_max, Hkv, d)
        self.k = [torch.zeros(shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        self.v = [torch.zeros(shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        self.cur = 0
        self.pk = to_dev(pr["prompt_k"]) if pr["prompt_k"].shape[0] else torch.zeros((1, Hkv, d), dtype=torch.bfloat16, device="cuda")[:0]
        self.pv = to_dev(pr["prompt_v"]) if pr["prompt_v"].shape[0] else torch.zeros((1, Hkv, d), dtype=torch.bfloat16, device="cuda")[:0]
        self.cu = i32_dev(pr["cu_prompt"])

    def step(self, s, dev_status=None, parent=None):
        import torch
        pr = self.pr
        src, dst = self.cur, 1 - self.cur
        par = i32_dev(pr["parent"][s] if parent is None else parent)
        bg.bg_beam_suffix_reorder(self.k[src], self.v[src], self.k[dst], self.v[dst], par, s,
                                  new_k=to_dev(pr["new_k"][s]), new_v=to_dev(pr["new_v"][s]), dev_status=dev_status)
        self.cur = dst
        q = to_dev(pr["q"][s])
        out = torch.empty_like(q)
        bg.bg_beam_decode_attn(q, self.pk, self.pv, self.cu, pr["max_prompt_len"], self.k[dst], self.v[dst], s + 1,
                               out, dev_status=dev_status)
        torch.cuda.synchronize()
        return out


def run_and_check(pr, suffix_max=None, requests=None, what=""):
    """Runs every step on the GPU; checks the reordered suffix bit-exactly and
    the attention output against the oracle (optionally on a subset of
    requests, which are independent)."""
    R, W, d = pr["R"], pr["W"], pr["head_dim"]
    steps = pr["steps"]
    gb = GpuBeams(pr, suffix_max or steps)
    hist = oracle.BeamHistory(R, W)
    scale = 1.0 / math.sqrt(d)
    reqs = list(range(R)) if requests is None else list(requests)
    cu = pr["cu_prompt"]
    pidx = np.concatenate([np.arange(cu[r], cu[r + 1]) for r in reqs]) if reqs else np.zeros(0, int)
    sub_cu = wl.cu_from_lengths([int(cu[r + 1] - cu[r]) for r in reqs])
    worst = (0.0, 0.0)
    for s in range(steps):
        out = gb.step(s)
        hist.step(pr["parent"][s], pr["new_k"][s], pr["new_v"][s])
        hk, hv = hist.materialise(pr["Hkv"], d)
        gk = bits_from_dev(gb.k[gb.cur])[:, :, :s + 1]
        gv = bits_from_dev(gb.v[gb.cur])[:, :, :s + 1]
        np.testing.assert_array_equal(gk, hk)
        np.testing.assert_array_equal(gv, hv)
        ref = oracle.decode(pr["q"][s][reqs], pr["prompt_k"][pidx], pr["prompt_v"][pidx], sub_cu, hk[reqs], hv[reqs],
                            scale)
        ma, rr = assert_parity(from_dev(out)[reqs], ref, f"{what} step {s}")
        worst = (max(worst[0], ma), max(worst[1], rr))
    return worst


@pytest.mark.parametrize("Hq,Hkv,d", [(14, 2, 64), (14, 2, 128), (4, 4, 64), (32, 2, 64), (16, 1, 128)])
def test_decode_small_parity(Hq, Hkv, d):
    pr = wl.make_decode_problem(3, 37, 4, Hq, Hkv, d, [130, 0, 257])
    run_and_check(pr, what=f"small Hq{Hq} Hkv{Hkv} d{d}")


def test_decode_short_prompt_config_full():
    cfg = wl.DECODE_CONFIGS["beam_short"]
    run_and_check(wl.make_decode_config_problem(cfg), what="beam_short")


def test_decode_long_prompt_config_sampled():
    cfg = wl.DECODE_CONFIGS["beam_long"]
    run_and_check(wl.make_decode_config_problem(cfg), requests=[0, 7, 15], what="beam_long")


def test_decode_prompt_only_and_suffix_only():
    import torch
    pr = wl.make_decode_problem(2, 9, 1, 14, 2, 64, [200, 0])
    gb = GpuBeams(pr, 2)
    # prompt only (suffix_len 0) is valid for request 0 and an empty row for request 1
    q = to_dev(pr["q"][0])
    out = torch.zeros_like(q)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.bg_beam_decode_attn(q, gb.pk, gb.pv, gb.cu, pr["max_prompt_len"], gb.k[0], gb.v[0], 0, out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bg.BG_DEVSTAT_EMPTY_ROW
    empty = np.zeros((2, 9, 0, 2, 64), np.uint16)
    ref = oracle.decode(pr["q"][0][:1], pr["prompt_k"], pr["prompt_v"], np.array([0, 200], np.int32), empty[:1],
                        empty[:1], 1 / 8)
    assert_parity(from_dev(out)[:1], ref, "prompt only")
    assert np.all(bits_from_dev(out)[1] == 0)          # the empty request was skipped
    # suffix only (request 1 has no prompt) after one step
    out2 = gb.step(0)
    hist = oracle.BeamHistory(2, 9)
    hist.step(pr["parent"][0], pr["new_k"][0], pr["new_v"][0])
    hk, hv = hist.materialise(2, 64)
    ref2 = oracle.decode(pr["q"][0], pr["prompt_k"], pr["prompt_v"], pr["cu_prompt"], hk, hv, 1 / 8)
    assert_parity(from_dev(out2), ref2, "suffix only")
    # a single key (no prompt, one suffix token) returns that value row exactly
    got = bits_from_dev(out2)[1]
    for h in range(14):
        np.testing.assert_array_equal(got[:, h], pr["new_v"][0][1][:, h // 7])


def test_decode_deterministic():
    pr = wl.make_decode_problem(2, 50, 2, 14, 2, 64, [300, 129])
    a = GpuBeams(pr, 2)
    b = GpuBeams(pr, 2)
    for s in range(2):
        oa, ob = a.step(s), b.step(s)
        np.testing.assert_array_equal(bits_from_dev(oa), bits_from_dev(ob))


def test_bad_parent_and_bad_cu_prompt_reported():
    import torch
    pr = wl.make_decode_problem(2, 8, 2, 14, 2, 64, [20, 30])
    gb = GpuBeams(pr, 2)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_parent = pr["parent"][0].copy()
    bad_parent[1, 3] = 8
    gb.step(0, dev_status=st, parent=bad_parent)
    assert int(st.item()) & bg.BG_DEVSTAT_PARENT
    st.zero_()
    gb.cu = i32_dev(np.array([0, 40, 50], np.int32))     # prompt 0 longer than max_prompt_len
    q = to_dev(pr["q"][1])
    out = torch.zeros_like(q)
    bg.bg_beam_decode_attn(q, gb.pk, gb.pv, gb.cu, pr["max_prompt_len"], gb.k[gb.cur], gb.v[gb.cur], 1, out,
                           dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & bg.BG_DEVSTAT_CU_PROMPT
    assert np.all(bits_from_dev(out)[0] == 0)
