"""bg_beam_select on the GPU against the fp64 selection oracle
(oracle/beam_select.py; section 1.1 of the page: local candidates per beam,
merged with accumulated scores, W kept, parent index out).

The kernel scores in fp32, the oracle in fp64, so two candidates whose scores
differ by less than the fp32 rounding may come out in either order.  What is
unique is compared exactly: the kept scores (sorted) within SCORE_TOL, and the
(parent, token) of every kept position whose oracle score is separated from
its neighbours (and from the first dropped score) by more than 2 * SCORE_TOL.
The rest is checked for validity: each kept pair is a real candidate whose
oracle score matches the kernel's score, pairs are distinct, scores are sorted.
Cases built with exactly equal scores compare the whole order exactly."""
import numpy as np
import pytest

from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from oracle import beam_select as ob

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-4     # fp32 logsumexp over up to 2^22 logits and fp32 sums of scores of size ~20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def run_gpu(logits: np.ndarray, cum: np.ndarray):
    import torch
    R, W, V = logits.shape
    lt = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    ct = torch.from_numpy(np.ascontiguousarray(cum, dtype=np.float32)).cuda()
    tok = torch.full((R, W), -7, dtype=torch.int32, device="cuda")
    par = torch.full((R, W), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((R, W), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(bg.bg_beam_select_workspace_size(R, W, V), dtype=torch.uint8, device="cuda")
    bg.bg_beam_select(lt, ct, tok, par, sc, workspace=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), par.cpu().numpy(), sc.cpu().numpy().astype(np.float64)


def check_against_oracle(logits, cum, exact_order=False):
    x = np.asarray(logits, dtype=np.float32)
    c = np.asarray(cum, dtype=np.float32)
    R, W, V = x.shape
    g_tok, g_par, g_sc = run_gpu(x, c)
    o_tok, o_par, o_sc = ob.beam_select(x, c)          # the same fp32 inputs, widened exactly
    lp = ob.log_softmax_rows(x)
    for r in range(R):
        assert np.all((g_par[r] >= 0) & (g_par[r] < W)) and np.all((g_tok[r] >= 0) & (g_tok[r] < V))
        assert len(set(zip(g_par[r].tolist(), g_tok[r].tolist()))) == W, "kept pairs must be distinct"
        s_of = c[r, g_par[r]].astype(np.float64) + lp[r, g_par[r], g_tok[r]]
        fin = np.isfinite(s_of)
        assert np.all(np.isfinite(g_sc[r]) == fin)
        assert np.max(np.abs(g_sc[r][fin] - s_of[fin]), initial=0.0) <= SCORE_TOL, "kernel score of a kept pair"
        assert np.all(np.diff(g_sc[r][fin]) <= SCORE_TOL), "kept candidates must be best first"
        # the kept scores are unique (as a sorted list) up to rounding
        o_fin = np.isfinite(o_sc[r])
        assert int(o_fin.sum()) == int(fin.sum())
        assert np.max(np.abs(np.sort(s_of[fin]) - np.sort(o_sc[r][o_fin])), initial=0.0) <= SCORE_TOL
        if exact_order:
            assert np.array_equal(g_tok[r], o_tok[r]) and np.array_equal(g_par[r], o_par[r])
            continue
        # positions the oracle decides by more than the rounding: same pair
        all_s = np.sort((c[r][:, None].astype(np.float64) + lp[r]).reshape(-1))[::-1]
        nxt = all_s[W] if all_s.size > W else -np.inf
        s = o_sc[r]
        for k in range(W):
            lo = s[k + 1] if k + 1 < W else nxt
            hi = s[k - 1] if k > 0 else np.inf
            if np.isfinite(s[k]) and s[k] - lo > 2 * SCORE_TOL and hi - s[k] > 2 * SCORE_TOL:
                assert (g_par[r, k], g_tok[r, k]) == (o_par[r, k], o_tok[r, k]), f"request {r} position {k}"


@pytest.mark.parametrize("R,W,V,sigma", [
    (2, 3, 5, 2.0), (3, 8, 1001, 3.0), (2, 16, 4096, 1.0), (4, 100, 65536, 3.0), (2, 400, 32768, 3.0),
    (1, 512, 8192, 0.5),
])
def test_select_random(R, W, V, sigma):
    rng = np.random.default_rng(R * 7919 + W * 31 + V)
    logits = rng.normal(0, sigma, size=(R, W, V)).astype(np.float32)
    cum = rng.normal(-3, 1, size=(R, W)).astype(np.float32)
    check_against_oracle(logits, cum)


def test_select_first_step():
    # only beam 0 alive: its W best tokens, parent 0 throughout
    rng = np.random.default_rng(21)
    R, W, V = 3, 100, 20000
    logits = rng.normal(0, 3, size=(R, W, V)).astype(np.float32)
    cum = np.full((R, W), -np.inf, dtype=np.float32)
    cum[:, 0] = 0.0
    g_tok, g_par, _ = run_gpu(logits, cum)
    assert np.all(g_par == 0)
    check_against_oracle(logits, cum)


def test_select_equal_logits_exact_ties():
    # every logit equal: every beam's scores tie exactly (the same arithmetic on the same
    # values, in fp32 and in fp64), so the order is fixed by the flat index alone; 8192 equal
    # keys in a row force the last radix level
    R, W, V = 2, 64, 8192
    logits = np.full((R, W, V), 2.5, dtype=np.float32)
    cum = np.zeros((R, W), dtype=np.float32)
    cum[1] = -np.arange(W, dtype=np.float32)                 # request 1: beam 0 best, then beam 1, ...
    check_against_oracle(logits, cum, exact_order=True)
    g_tok, g_par, _ = run_gpu(logits, cum)
    assert np.array_equal(g_par[0], np.zeros(W)) and np.array_equal(g_tok[0], np.arange(W))


def test_select_duplicate_beams_tie_by_parent():
    # two beams with identical logits and scores: equal candidates keep the smaller parent first
    rng = np.random.default_rng(23)
    R, W, V = 2, 8, 3000
    base = rng.normal(0, 2, size=(R, 1, V)).astype(np.float32)
    logits = np.repeat(base, W, axis=1)
    cum = np.zeros((R, W), dtype=np.float32)
    check_against_oracle(logits, cum, exact_order=True)


def test_select_dead_beams_never_kept():
    rng = np.random.default_rng(24)
    R, W, V = 2, 50, 5000
    logits = rng.normal(0, 3, size=(R, W, V)).astype(np.float32)
    cum = rng.normal(-2, 1, size=(R, W)).astype(np.float32)
    cum[:, ::3] = -np.inf
    g_tok, g_par, g_sc = run_gpu(logits, cum)
    assert np.all(g_par % 3 != 0) and np.all(np.isfinite(g_sc))
    check_against_oracle(logits, cum)


def test_select_deterministic():
    rng = np.random.default_rng(25)
    logits = rng.normal(0, 3, size=(4, 100, 30000)).astype(np.float32)
    cum = rng.normal(-3, 1, size=(4, 100)).astype(np.float32)
    a = run_gpu(logits, cum)
    b = run_gpu(logits, cum)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("order", ["ascending", "descending"])
def test_select_sorted_rows(order):
    # ascending logits: every block of the row beats everything before it, so the row
    # kernel's filter never settles and its buffer compacts again and again; descending:
    # the first block holds the winners and the filter drops the rest at once
    R, W, V = 2, 512, 65536
    rng = np.random.default_rng(26)
    ramp = np.arange(V, dtype=np.float64) * 1e-3
    if order == "descending":
        ramp = ramp[::-1]
    logits = np.broadcast_to((ramp - 30.0).astype(np.float32), (R, W, V)).copy()
    logits += rng.normal(0, 1e-2, size=(R, W, 1)).astype(np.float32)   # beams differ by a shift
    cum = rng.normal(-3, 1, size=(R, W)).astype(np.float32)
    check_against_oracle(logits, cum)


def test_select_masked_vocab_ties_at_minus_inf():
    # one finite logit per beam (the rest masked to -inf) and half the beams dead: fewer
    # finite candidates than W, so the kept list ends in -inf scores ordered by the flat
    # index b * V + v alone; every row ties at -inf far beyond what one gather holds
    R, W, V = 2, 64, 10001
    rng = np.random.default_rng(27)
    logits = np.full((R, W, V), -np.inf, dtype=np.float32)
    pos = rng.integers(0, V, size=(R, W))
    for r in range(R):
        for b in range(W):
            logits[r, b, pos[r, b]] = rng.normal(0, 3)
    cum = rng.normal(-3, 1, size=(R, W)).astype(np.float32)
    cum[:, 1::2] = -np.inf
    check_against_oracle(logits, cum, exact_order=True)


@pytest.mark.parametrize("V", [20000, 20001])
def test_select_quantised_logits_ties(V):
    # logits on a grid of 0.5: the W-th best value is shared by dozens of tokens, so the
    # selection resolves ties by token inside the gathered set; one live beam keeps every
    # score exact in fp32 and fp64, so the whole order is compared
    R, W = 2, 64
    rng = np.random.default_rng(28 + V)
    logits = (np.round(rng.normal(0, 3, size=(R, W, V)) * 2) / 2).astype(np.float32)
    cum = np.full((R, W), -np.inf, dtype=np.float32)
    cum[:, 0] = 0.0
    check_against_oracle(logits, cum, exact_order=True)


@pytest.mark.parametrize("V", [131072, 131077])
def test_select_large_vocab(V):
    # 131,072 logits is the largest row whose group maxima stay in shared memory for the second
    # pass; one more float4 group (131,077) takes the path that streams the row again
    R, W = 2, 48
    rng = np.random.default_rng(29 + V)
    logits = rng.normal(0, 3, size=(R, W, V)).astype(np.float32)
    cum = rng.normal(-3, 1, size=(R, W)).astype(np.float32)
    check_against_oracle(logits, cum)


def test_select_many_requests_wide_beams():
    # 24 requests at beam 512: 13 level-1 slices per request, whose 40 x 512 candidate keys are
    # too many to keep in shared memory, so level 1 recomputes them in every pass
    R, W, V = 24, 512, 600
    rng = np.random.default_rng(30)
    logits = rng.normal(0, 2, size=(R, W, V)).astype(np.float32)
    cum = rng.normal(-3, 1, size=(R, W)).astype(np.float32)
    check_against_oracle(logits, cum)
