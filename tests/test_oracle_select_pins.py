"""Pins of the beam candidate selection oracle (oracle/beam_select.py) to
things other than itself: closed forms, invariants of the softmax, the first
step and greedy special cases, and brute force on tiny inputs.

Page: "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.1 (each step:
local candidates per beam's token distribution, merged with accumulated
scores, W kept; candidates, scores and parent index come out).

Every check takes the oracle module as an argument so that
test_oracle_select_mutations.py can run the same checks on copies of the oracle
with planted mistakes."""
import math

import numpy as np
import pytest

from oracle import beam_select as bs_real


def check_two_token_closed_form(bs):
    # two beams, two tokens: log p(v | b) = -log(1 + exp(x_other - x_v))
    x = np.array([[[0.3, -1.1], [2.0, 1.5]]])
    cum = np.array([[-0.2, -1.9]])
    cand = []
    for b in range(2):
        for v in range(2):
            lp = -math.log1p(math.exp(x[0, b, 1 - v] - x[0, b, v]))
            cand.append((cum[0, b] + lp, b, v))
    best = sorted(cand, key=lambda c: (-c[0], c[1] * 2 + c[2]))[:2]
    tok, par, sc = bs.beam_select(x, cum)
    assert [int(t) for t in tok[0]] == [c[2] for c in best]
    assert [int(p) for p in par[0]] == [c[1] for c in best]
    assert np.allclose(sc[0], [c[0] for c in best], rtol=0, atol=1e-12)


def check_brute_force(bs):
    rng = np.random.default_rng(11)
    R, W, V = 2, 3, 5
    x = rng.normal(0, 2, size=(R, W, V))
    cum = rng.normal(0, 1, size=(R, W))
    tok, par, sc = bs.beam_select(x, cum)
    for r in range(R):
        s = []
        for b in range(W):
            m = max(x[r, b])
            lse = m + math.log(sum(math.exp(float(t) - m) for t in x[r, b]))
            for v in range(V):
                s.append(float(cum[r, b]) + float(x[r, b, v]) - lse)
        keep = sorted(range(W * V), key=lambda i: (-s[i], i))[:W]
        assert [int(t) for t in tok[r]] == [i % V for i in keep]
        assert [int(p) for p in par[r]] == [i // V for i in keep]
        assert np.allclose(sc[r], [s[i] for i in keep], rtol=0, atol=1e-12)


def check_shift_invariance(bs):
    # softmax does not see a constant added to all logits of one beam
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, size=(3, 4, 50))
    cum = rng.normal(0, 1, size=(3, 4))
    shift = rng.normal(0, 10, size=(3, 4, 1))
    a = bs.beam_select(x, cum)
    b = bs.beam_select(x + shift, cum)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.allclose(a[2], b[2], rtol=0, atol=1e-9)


def check_greedy_single_beam(bs):
    # W = 1: the best token of the one beam, score = cum + max - logsumexp
    rng = np.random.default_rng(13)
    x = rng.normal(0, 1, size=(4, 1, 37))
    cum = rng.normal(0, 1, size=(4, 1))
    tok, par, sc = bs.beam_select(x, cum)
    for r in range(4):
        v = int(np.argmax(x[r, 0]))
        lse = math.log(sum(math.exp(float(t)) for t in x[r, 0]))
        assert int(tok[r, 0]) == v and int(par[r, 0]) == 0
        assert abs(sc[r, 0] - (cum[r, 0] + x[r, 0, v] - lse)) < 1e-12


def check_first_step(bs):
    # only beam 0 alive: its W best tokens, all with parent 0, best first
    rng = np.random.default_rng(14)
    W, V = 6, 40
    x = rng.normal(0, 1, size=(2, W, V))
    cum = np.full((2, W), -np.inf)
    cum[:, 0] = 0.0
    tok, par, sc = bs.beam_select(x, cum)
    for r in range(2):
        want = sorted(range(V), key=lambda v: -x[r, 0, v])[:W]
        assert [int(t) for t in tok[r]] == want
        assert np.all(par[r] == 0)
        assert np.all(np.diff(sc[r]) <= 0)


def check_uniform_rows_tie_order(bs):
    # equal logits in a beam: every token has log p = -log V; equal scores keep the
    # smaller flat index first
    V = 4
    x = np.zeros((1, 3, V))
    x[0, 1] = 5.0                                   # constant rows: the value does not matter
    cum = np.array([[0.0, -0.5, -1.0]])
    tok, par, sc = bs.beam_select(x, cum)
    assert [int(t) for t in tok[0]] == [0, 1, 2]
    assert [int(p) for p in par[0]] == [0, 0, 0]
    assert np.allclose(sc[0], -math.log(V), rtol=0, atol=1e-15)
    cum2 = np.zeros((1, 3))                        # all scores equal: the first W flat indices
    tok, par, _ = bs.beam_select(x, cum2)
    assert [int(t) for t in tok[0]] == [0, 1, 2] and [int(p) for p in par[0]] == [0, 0, 0]


def check_probabilities_sum_to_one(bs):
    # one live beam and W = V: all of its tokens are kept; exp(score - cum) sums to 1
    rng = np.random.default_rng(15)
    V = 9
    x = rng.normal(0, 3, size=(1, V, V))
    cum = np.full((1, V), -np.inf)
    cum[0, 0] = -2.5
    tok, par, sc = bs.beam_select(x, cum)
    assert sorted(int(t) for t in tok[0]) == list(range(V))
    assert abs(sum(math.exp(float(s) + 2.5) for s in sc[0]) - 1.0) < 1e-12


def check_output_structure(bs):
    rng = np.random.default_rng(16)
    R, W, V = 3, 8, 30
    x = rng.normal(0, 1, size=(R, W, V))
    cum = rng.normal(0, 1, size=(R, W))
    tok, par, sc = bs.beam_select(x, cum)
    for r in range(R):
        assert np.all(np.diff(sc[r]) <= 0)
        pairs = set(zip(par[r].tolist(), tok[r].tolist()))
        assert len(pairs) == W
        assert all(0 <= p < W and 0 <= t < V for p, t in pairs)


CHECKS = [check_two_token_closed_form, check_brute_force, check_shift_invariance, check_greedy_single_beam,
          check_first_step, check_uniform_rows_tie_order, check_probabilities_sum_to_one, check_output_structure]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_select_oracle_pin(check):
    check(bs_real)
