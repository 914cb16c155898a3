"""GPU parity of a whole decode step through the C ABI (bg_beam_decode_step).

The call reorders each beam's suffix by the parent index, appends the step's
token and attends over [shared prompt ; the beam's suffix].  It is checked
three ways on the same seeded inputs:
  * the suffix it leaves in dst equals the oracle's explicit per-beam histories
    bit for bit;
  * the output matches the fp64 oracle within the decode tolerance;
  * output and suffix are bit-identical to the two separate calls
    (bg_beam_suffix_reorder, then bg_beam_decode_attn).
Both suffix buffers start as bf16 NaN, so a row read before it was written
would poison the output."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu

BF16_NAN = 0x7FC0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


class Beams:
    """Device state of one beam search: ping-pong suffix buffers filled with NaN; `one_call`
    selects one bg_beam_decode_step per step or the separate reorder and attention calls."""

    def __init__(self, pr, suffix_max, one_call=True):
        import torch
        R, W, Hkv, d = pr["R"], pr["W"], pr["Hkv"], pr["head_dim"]
        self.pr, self.one_call = pr, one_call
        shape = (R, W, suffix_max, Hkv, d)
        nan = np.full(shape, BF16_NAN, np.uint16)
        self.k = [to_dev(nan) for _ in range(2)]
        self.v = [to_dev(nan) for _ in range(2)]
        self.cur = 0
        empty = torch.zeros((1, Hkv, d), dtype=torch.bfloat16, device="cuda")[:0]
        self.pk = to_dev(pr["prompt_k"]) if pr["prompt_k"].shape[0] else empty
        self.pv = to_dev(pr["prompt_v"]) if pr["prompt_v"].shape[0] else empty
        self.cu = i32_dev(pr["cu_prompt"])

    def step(self, s, dev_status=None, parent=None, src_at_first=False):
        import torch
        pr = self.pr
        src, dst = self.cur, 1 - self.cur
        par = i32_dev(pr["parent"][s] if parent is None else parent)
        nk, nv = to_dev(pr["new_k"][s]), to_dev(pr["new_v"][s])
        q = to_dev(pr["q"][s])
        out = torch.empty_like(q)
        if self.one_call:
            give_src = s > 0 or src_at_first
            bg.bg_beam_decode_step(q, self.pk, self.pv, self.cu, pr["max_prompt_len"],
                                   self.k[src] if give_src else None, self.v[src] if give_src else None, par, nk, nv,
                                   self.k[dst], self.v[dst], s + 1, out, dev_status=dev_status)
        else:
            bg.bg_beam_suffix_reorder(self.k[src], self.v[src], self.k[dst], self.v[dst], par, s, new_k=nk, new_v=nv,
                                      dev_status=dev_status)
            bg.bg_beam_decode_attn(q, self.pk, self.pv, self.cu, pr["max_prompt_len"], self.k[dst], self.v[dst], s + 1,
                                   out, dev_status=dev_status)
        torch.cuda.synchronize()
        self.cur = dst
        return out


def run_and_check(pr, suffix_max=None, requests=None, what="", against_two_call=True):
    R, W, d = pr["R"], pr["W"], pr["head_dim"]
    steps = pr["steps"]
    S = suffix_max or steps
    one = Beams(pr, S, one_call=True)
    pair = Beams(pr, S, one_call=False) if against_two_call else None
    hist = oracle.BeamHistory(R, W)
    scale = 1.0 / math.sqrt(d)
    reqs = list(range(R)) if requests is None else list(requests)
    cu = pr["cu_prompt"]
    pidx = np.concatenate([np.arange(cu[r], cu[r + 1]) for r in reqs]) if reqs else np.zeros(0, int)
    sub_cu = wl.cu_from_lengths([int(cu[r + 1] - cu[r]) for r in reqs])
    for s in range(steps):
        out = one.step(s)
        hist.step(pr["parent"][s], pr["new_k"][s], pr["new_v"][s])
        hk, hv = hist.materialise(pr["Hkv"], d)
        gk = bits_from_dev(one.k[one.cur])[:, :, :s + 1]
        gv = bits_from_dev(one.v[one.cur])[:, :, :s + 1]
        np.testing.assert_array_equal(gk, hk, err_msg=f"{what} step {s}: suffix K")
        np.testing.assert_array_equal(gv, hv, err_msg=f"{what} step {s}: suffix V")
        ref = oracle.decode(pr["q"][s][reqs], pr["prompt_k"][pidx], pr["prompt_v"][pidx], sub_cu, hk[reqs], hv[reqs],
                            scale)
        assert_parity(from_dev(out)[reqs], ref, f"{what} step {s}")
        if pair is not None:
            out2 = pair.step(s)
            np.testing.assert_array_equal(bits_from_dev(out), bits_from_dev(out2),
                                          err_msg=f"{what} step {s}: one call vs two calls")
            np.testing.assert_array_equal(bits_from_dev(one.k[one.cur])[:, :, :s + 1],
                                          bits_from_dev(pair.k[pair.cur])[:, :, :s + 1])
            np.testing.assert_array_equal(bits_from_dev(one.v[one.cur])[:, :, :s + 1],
                                          bits_from_dev(pair.v[pair.cur])[:, :, :s + 1])


@pytest.mark.parametrize("Hq,Hkv,d", [(14, 2, 64), (14, 2, 128), (4, 4, 64), (32, 2, 64), (16, 1, 128),
                                      (7, 1, 64), (64, 1, 64)])
def test_step_small_parity(Hq, Hkv, d):
    # W = 37 is not a multiple of the beams per tile: items end mid-tile, and the last suffix
    # tile of a request's last item reaches into the next request's beams
    pr = wl.make_decode_problem(3, 37, 4, Hq, Hkv, d, [130, 0, 257])
    run_and_check(pr, what=f"step Hq{Hq} Hkv{Hkv} d{d}")


def test_step_long_suffix():
    # t up to BG_MAX_SUFFIX: four beams per suffix tile, many (beam, slot) rows per item
    pr = wl.make_decode_problem(2, 11, bg.BG_MAX_SUFFIX, 14, 2, 64, [70, 0])
    run_and_check(pr, suffix_max=bg.BG_MAX_SUFFIX, what="t up to 16")


def test_step_short_prompt_config_full():
    cfg = wl.DECODE_CONFIGS["beam_short"]
    run_and_check(wl.make_decode_config_problem(cfg), what="beam_short")


def test_step_long_prompt_config_sampled():
    cfg = wl.DECODE_CONFIGS["beam_long"]
    run_and_check(wl.make_decode_config_problem(cfg), requests=[0, 7, 15], what="beam_long")


def test_step_first_step_ignores_src():
    # at t = 1 nothing is moved: passing the (NaN) previous buffer or NULL gives the same result
    pr = wl.make_decode_problem(2, 20, 1, 14, 2, 64, [90, 33])
    a, b = Beams(pr, 3), Beams(pr, 3)
    oa = a.step(0)
    ob = b.step(0, src_at_first=True)
    np.testing.assert_array_equal(bits_from_dev(oa), bits_from_dev(ob))
    np.testing.assert_array_equal(bits_from_dev(a.k[a.cur]), bits_from_dev(b.k[b.cur]))


def test_step_deterministic():
    pr = wl.make_decode_problem(2, 50, 3, 14, 2, 64, [300, 129])
    a, b = Beams(pr, 3), Beams(pr, 3)
    for s in range(3):
        np.testing.assert_array_equal(bits_from_dev(a.step(s)), bits_from_dev(b.step(s)))


def test_step_bad_parent_reported():
    import torch
    pr = wl.make_decode_problem(2, 8, 2, 14, 2, 64, [20, 30])
    gb = Beams(pr, 2)
    gb.step(0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = pr["parent"][1].copy()
    bad[1, 3] = -1
    gb.step(1, dev_status=st, parent=bad)
    assert int(st.item()) & bg.BG_DEVSTAT_PARENT
    # every other beam still got its reordered suffix
    hist = oracle.BeamHistory(2, 8)
    hist.step(pr["parent"][0], pr["new_k"][0], pr["new_v"][0])
    good = bad.copy()
    good[1, 3] = 0
    hist.step(good, pr["new_k"][1], pr["new_v"][1])
    hk, _ = hist.materialise(2, 64)
    gk = bits_from_dev(gb.k[gb.cur])[:, :, :2]
    keep = np.ones((2, 8), bool)
    keep[1, 3] = False
    np.testing.assert_array_equal(gk[keep], hk[keep])
