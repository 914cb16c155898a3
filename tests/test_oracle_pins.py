"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, each chosen so that a plausible mistake in the oracle fails at least one.

Mistake -> test that catches it
  dropped / wrong scale ............ test_two_keys_closed_form, test_one_hot_v_weights_log_ratio
  causal off by one (j<p, j<=p+1) .. test_length_one_returns_own_v, test_uniform_prefix_mean_golden,
                                     test_causality_future_keys_do_not_matter
  k and v swapped / transposed ..... test_constant_v_returns_constant, test_uniform_prefix_mean_golden
  wrong GQA head mapping ........... test_gqa_equals_repeated_kv, test_one_hot_v_weights_log_ratio
  wrong sequence offsets ........... test_packed_equals_each_sequence_alone, test_permuting_sequences
  softmax not normalised ........... test_one_hot_v_weights_log_ratio (rows sum to 1)
  decode ignores prompt / suffix ... test_decode_equals_full_kv, test_decode_equals_last_prefill_row
  reorder gathers the wrong beam ... test_history_follows_parent_chain, test_history_composition
  last token off by one or head .... test_last_token_equals_last_padded_row, test_last_token_closed_forms
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from attention_packed_varlen_causal_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return wl.bf16_bits_from_f32(np.asarray(x, dtype=np.float32))


def widen(b):
    return wl.bf16_bits_to_f32(b).astype(np.float64)


def rand_prefill(lengths, Hq, Hkv, d, seed):
    return wl.make_prefill_inputs(lengths, Hq, Hkv, d, seeds=(seed, seed + 1, seed + 2))


# ---------------------------------------------------------------- closed forms
def test_uniform_prefix_mean_golden():
    fx = json.load(open(os.path.join(GOLDEN, "closed_form_fixtures.json")))["uniform_prefix_mean"]
    lengths, Hq, Hkv, d = fx["lengths"], fx["Hq"], fx["Hkv"], fx["head_dim"]
    T = sum(lengths)
    v_rows = [[Fraction(x).limit_denominator() for x in row] for row in fx["v"]]
    k = bits(np.array(fx["k"], dtype=np.float32).reshape(T, Hkv, d))
    v = bits(np.array(fx["v"], dtype=np.float32).reshape(T, Hkv, d))
    q = bits(np.zeros((T, Hq, d), dtype=np.float32))
    cu = wl.cu_from_lengths(lengths)
    out = oracle.prefill(q, k, v, cu, scale=0.7)
    for i, L in enumerate(lengths):
        s0 = int(cu[i])
        for p in range(L):
            expect = [sum(v_rows[s0 + j][c] for j in range(p + 1)) / (p + 1) for c in range(d)]
            for h in range(Hq):
                for c in range(d):
                    assert abs(out[s0 + p, h, c] - float(expect[c])) < 1e-14


def test_two_keys_closed_form():
    fx = json.load(open(os.path.join(GOLDEN, "closed_form_fixtures.json")))["two_keys"]
    d = fx["head_dim"]
    scale = 1.0 / math.sqrt(d)
    # one sequence of length 2; row 1 sees both keys
    q = bits(np.array([[fx["q"]], [fx["q"]]], dtype=np.float32))
    k = bits(np.array([[fx["k0"]], [fx["k1"]]], dtype=np.float32))
    v = bits(np.array([[fx["v0"]], [fx["v1"]]], dtype=np.float32))
    out, lse = oracle.prefill(q, k, v, np.array([0, 2], np.int32), scale, want_lse=True)
    z0 = scale * (fx["q"][0] * fx["k0"][0] + fx["q"][1] * fx["k0"][1])
    z1 = scale * (fx["q"][0] * fx["k1"][0] + fx["q"][1] * fx["k1"][1])
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))
    for c in range(d):
        expect = (1 - w1) * fx["v0"][c] + w1 * fx["v1"][c]
        assert abs(out[1, 0, c] - expect) < 1e-15
        assert out[0, 0, c] == fx["v0"][c]          # row 0 sees only key 0
    assert abs(lse[1, 0] - (max(z0, z1) + math.log1p(math.exp(-abs(z0 - z1))))) < 1e-15
    assert abs(lse[0, 0] - z0) < 1e-15


def test_length_one_returns_own_v():
    x = rand_prefill([1, 1, 1], 4, 2, 16, seed=11)
    out = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], 0.25)
    kv = widen(x["v"])
    for h in range(4):
        np.testing.assert_array_equal(out[:, h, :], kv[:, h // 2, :])


def test_constant_v_returns_constant():
    x = rand_prefill([5, 9, 2], 4, 2, 8, seed=21)
    c = np.linspace(-3, 3, 8, dtype=np.float32)
    v = bits(np.broadcast_to(c, x["v"].shape))
    out = oracle.prefill(x["q"], x["k"], v, x["cu_seqlens"], 1 / math.sqrt(8))
    assert np.max(np.abs(out - widen(bits(c))[None, None, :])) < 1e-14
    ones = bits(np.ones(x["v"].shape, np.float32))
    out1 = oracle.prefill(x["q"], x["k"], ones, x["cu_seqlens"], 1 / math.sqrt(8))
    assert np.max(np.abs(out1 - 1.0)) < 1e-15


def test_one_hot_v_weights_log_ratio():
    """V = one-hot rows exposes the softmax weights: rows sum to 1, are zero
    beyond the diagonal, and log(w_j / w_0) = scale * q.(k_j - k_0)."""
    L, Hq, Hkv, d = 7, 4, 2, 8
    x = rand_prefill([L], Hq, Hkv, d, seed=31)
    v = np.zeros((L, Hkv, d), np.float32)
    for j in range(L):
        v[j, :, j] = 1.0
    scale = 0.37
    out = oracle.prefill(x["q"], x["k"], bits(v), x["cu_seqlens"], scale)
    Q, K = widen(x["q"]), widen(x["k"])
    for p in range(L):
        for h in range(Hq):
            w = out[p, h]
            assert abs(w.sum() - 1.0) < 1e-13
            assert np.all(w[p + 1:] == 0.0)
            assert np.all(w[:p + 1] > 0.0)
            for j in range(1, p + 1):
                dz = scale * float(Q[p, h] @ (K[j, h // 2] - K[0, h // 2]))
                assert abs(math.log(w[j] / w[0]) - dz) < 1e-10


# ---------------------------------------------------------------- invariants
def test_causality_future_keys_do_not_matter():
    x = rand_prefill([12], 2, 1, 16, seed=41)
    scale = 0.25
    base = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    p = 5
    k2, v2 = x["k"].copy(), x["v"].copy()
    k2[p + 1:] = bits(widen(k2[p + 1:]) * -3 + 1)
    v2[p + 1:] = bits(widen(v2[p + 1:]) * 2 - 5)
    pert = oracle.prefill(x["q"], k2, v2, x["cu_seqlens"], scale)
    np.testing.assert_array_equal(pert[:p + 1], base[:p + 1])
    assert np.max(np.abs(pert[p + 1:] - base[p + 1:])) > 1e-3
    # perturbing key p itself must change row p (the diagonal is attended)
    v3 = x["v"].copy()
    v3[p] = bits(widen(v3[p]) + 4)
    pert3 = oracle.prefill(x["q"], x["k"], v3, x["cu_seqlens"], scale)
    np.testing.assert_array_equal(pert3[:p], base[:p])
    assert np.max(np.abs(pert3[p] - base[p])) > 1e-3


def test_packed_equals_each_sequence_alone():
    lengths = [3, 17, 1, 40, 9]
    x = rand_prefill(lengths, 4, 2, 16, seed=51)
    scale = 0.25
    packed = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    cu = x["cu_seqlens"]
    for i in range(len(lengths)):
        a, b = int(cu[i]), int(cu[i + 1])
        alone = oracle.prefill(x["q"][a:b], x["k"][a:b], x["v"][a:b], np.array([0, b - a], np.int32), scale)
        np.testing.assert_array_equal(packed[a:b], alone)


def test_packed_equals_padded_masked_numpy():
    lengths = [3, 17, 1, 40, 9, 0, 23]
    x = rand_prefill(lengths, 6, 2, 32, seed=61)
    scale = 1 / math.sqrt(32)
    a = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    b = oracle_np.prefill_padded(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    assert np.max(np.abs(a - b)) < 1e-12


def test_permuting_sequences_permutes_outputs():
    lengths = [5, 11, 2, 8]
    x = rand_prefill(lengths, 4, 4, 8, seed=71)
    cu = x["cu_seqlens"]
    scale = 0.3
    base = oracle.prefill(x["q"], x["k"], x["v"], cu, scale)
    perm = [2, 0, 3, 1]
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in perm])
    cu2 = wl.cu_from_lengths([lengths[i] for i in perm])
    out2 = oracle.prefill(x["q"][idx], x["k"][idx], x["v"][idx], cu2, scale)
    np.testing.assert_array_equal(out2, base[idx])


def test_gqa_equals_repeated_kv():
    lengths = [6, 13]
    Hq, Hkv, d = 6, 2, 8
    x = rand_prefill(lengths, Hq, Hkv, d, seed=81)
    scale = 0.35
    gqa = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    k_rep = np.repeat(x["k"], Hq // Hkv, axis=1)
    v_rep = np.repeat(x["v"], Hq // Hkv, axis=1)
    mha = oracle.prefill(x["q"], k_rep, v_rep, x["cu_seqlens"], scale)
    np.testing.assert_array_equal(gqa, mha)


def test_chunked_queries_equal_one_shot():
    """Chunked prefill (page 2, 分块 prefill): rows of a later chunk see all
    earlier chunks' keys through the cache.  Rebuilt with the decode oracle:
    earlier chunks act as the prompt, the chunk's own keys up to row p as the
    suffix."""
    L, Hq, Hkv, d, chunk = 13, 2, 1, 8, 4
    x = rand_prefill([L], Hq, Hkv, d, seed=91)
    scale = 0.3
    one_shot = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
    for a in range(0, L, chunk):
        for p in range(a, min(a + chunk, L)):
            t = p - a + 1
            q = x["q"][p].reshape(1, 1, Hq, d)
            hk = x["k"][a:p + 1].reshape(1, 1, t, Hkv, d)
            hv = x["v"][a:p + 1].reshape(1, 1, t, Hkv, d)
            o = oracle.decode(q, x["k"][:a], x["v"][:a], np.array([0, a], np.int32), hk, hv, scale)
            assert np.max(np.abs(o[0, 0] - one_shot[p])) < 1e-12


def _py_attention(qrow, keys, vals, scale):
    """Third implementation: scalar Python with the math module."""
    z = [scale * sum(a * b for a, b in zip(qrow, kk)) for kk in keys]
    m = max(z)
    w = [math.exp(zz - m) for zz in z]
    s = sum(w)
    return [sum(w[j] * vals[j][c] for j in range(len(keys))) / s for c in range(len(qrow))]


def test_brute_force_tiny():
    rng = np.random.default_rng(5)
    for trial in range(20):
        d = int(rng.integers(1, 5))
        Hkv = int(rng.integers(1, 3))
        g = int(rng.integers(1, 3))
        Hq = Hkv * g
        lengths = rng.integers(0, 6, size=int(rng.integers(1, 4))).tolist()
        x = rand_prefill(lengths, Hq, Hkv, d, seed=100 + trial)
        scale = float(rng.uniform(0.1, 2.0))
        out = oracle.prefill(x["q"], x["k"], x["v"], x["cu_seqlens"], scale)
        Q, K, V = widen(x["q"]).tolist(), widen(x["k"]).tolist(), widen(x["v"]).tolist()
        cu = x["cu_seqlens"]
        for i in range(len(lengths)):
            s0 = int(cu[i])
            for p in range(lengths[i]):
                for h in range(Hq):
                    kh = h // g
                    ref = _py_attention(Q[s0 + p][h], [K[s0 + j][kh] for j in range(p + 1)],
                                        [V[s0 + j][kh] for j in range(p + 1)], scale)
                    assert np.max(np.abs(out[s0 + p, h] - np.array(ref))) < 1e-12


def test_oracle_rejects_invalid():
    x = rand_prefill([3, 4], 2, 1, 4, seed=3)
    with pytest.raises(ValueError):
        oracle.prefill(x["q"], x["k"], x["v"], np.array([0, 5, 7], np.int32)[[0, 2, 1]], 1.0)
    with pytest.raises(ValueError):
        oracle.decode(np.zeros((1, 1, 2, 4), np.uint16), x["k"][:0], x["v"][:0], np.array([0, 0], np.int32),
                      np.zeros((1, 1, 0, 1, 4), np.uint16), np.zeros((1, 1, 0, 1, 4), np.uint16), 1.0)


# ---------------------------------------------------------------- decode
def _decode_problem(R, W, steps, Hq, Hkv, d, prompts, layer=0):
    return wl.make_decode_problem(R, W, steps, Hq, Hkv, d, prompts, layer=layer)


def test_decode_equals_full_kv():
    R, W, steps, Hq, Hkv, d = 3, 5, 3, 6, 2, 16
    pr = _decode_problem(R, W, steps, Hq, Hkv, d, [7, 0, 12])
    scale = 1 / math.sqrt(d)
    hist = oracle.BeamHistory(R, W)
    cu = pr["cu_prompt"]
    for s in range(steps):
        hist.step(pr["parent"][s], pr["new_k"][s], pr["new_v"][s])
        hk, hv = hist.materialise(Hkv, d)
        out = oracle.decode(pr["q"][s], pr["prompt_k"], pr["prompt_v"], cu, hk, hv, scale)
        for r in range(R):
            for b in range(W):
                keys = np.concatenate([pr["prompt_k"][cu[r]:cu[r + 1]], hk[r, b]], axis=0)
                vals = np.concatenate([pr["prompt_v"][cu[r]:cu[r + 1]], hv[r, b]], axis=0)
                ref = oracle_np.full_kv_attention(pr["q"][s][r, b][None], keys, vals, scale)[0]
                assert np.max(np.abs(out[r, b] - ref)) < 1e-12


def test_decode_equals_last_prefill_row():
    """Cross-mode: decoding beam b equals the last row of causal prefill over
    the materialised sequence prompt_r ++ suffix(r, b) (section 1.2: the
    shared prompt K/V is the same for every beam)."""
    R, W, steps, Hq, Hkv, d = 2, 4, 4, 4, 2, 8
    pr = _decode_problem(R, W, steps, Hq, Hkv, d, [9, 3])
    scale = 0.4
    hist = oracle.BeamHistory(R, W)
    cu = pr["cu_prompt"]
    rng = np.random.default_rng(123)
    for s in range(steps):
        hist.step(pr["parent"][s], pr["new_k"][s], pr["new_v"][s])
        hk, hv = hist.materialise(Hkv, d)
        out = oracle.decode(pr["q"][s], pr["prompt_k"], pr["prompt_v"], cu, hk, hv, scale)
        for r in range(R):
            for b in range(W):
                ks = np.concatenate([pr["prompt_k"][cu[r]:cu[r + 1]], hk[r, b]], axis=0)
                vs = np.concatenate([pr["prompt_v"][cu[r]:cu[r + 1]], hv[r, b]], axis=0)
                n = ks.shape[0]
                qs = bits(rng.standard_normal((n, Hq, d)).astype(np.float32))
                qs[-1] = pr["q"][s][r, b]
                full = oracle.prefill(qs, ks, vs, np.array([0, n], np.int32), scale)
                assert np.max(np.abs(full[-1] - out[r, b])) < 1e-12


def test_decode_empty_prompt_single_suffix_returns_v():
    R, W, Hq, Hkv, d = 2, 3, 4, 2, 8
    pr = _decode_problem(R, W, 1, Hq, Hkv, d, [0, 0])
    hist = oracle.BeamHistory(R, W)
    hist.step(pr["parent"][0], pr["new_k"][0], pr["new_v"][0])
    hk, hv = hist.materialise(Hkv, d)
    out = oracle.decode(pr["q"][0], pr["prompt_k"], pr["prompt_v"], pr["cu_prompt"], hk, hv, 0.5)
    for h in range(Hq):
        np.testing.assert_array_equal(out[:, :, h, :], widen(pr["new_v"][0][:, :, h // 2, :]))


def test_history_follows_parent_chain():
    R, W, steps = 2, 6, 5
    rng = np.random.default_rng(9)
    hist = oracle.BeamHistory(R, W)
    parents, tokens = [], []
    for s in range(steps):
        par = rng.integers(0, W, size=(R, W)).astype(np.int32)
        tok = np.arange(R * W, dtype=np.uint16).reshape(R, W, 1, 1) + np.uint16(100 * s)
        hist.step(par, tok, tok)
        parents.append(par)
        tokens.append(tok)
    hk, _ = hist.materialise(1, 1)
    # trace each final beam backwards through its ancestors
    for r in range(R):
        for b in range(W):
            chain = []
            cur = b
            for s in reversed(range(steps)):
                chain.append(int(tokens[s][r, cur, 0, 0]))
                cur = int(parents[s][r, cur])
            assert hk[r, b, :, 0, 0].tolist() == chain[::-1]


def test_history_identity_and_composition():
    R, W = 2, 5
    rng = np.random.default_rng(10)
    h = oracle.BeamHistory(R, W)
    for s in range(3):
        tok = rng.integers(0, 60000, size=(R, W, 2, 3)).astype(np.uint16)
        h.step(rng.integers(0, W, size=(R, W)), tok, tok + 1)
    k0, v0 = h.materialise(2, 3)
    ident = np.tile(np.arange(W), (R, 1))
    h.step(ident)
    k1, v1 = h.materialise(2, 3)
    np.testing.assert_array_equal(k0, k1)
    np.testing.assert_array_equal(v0, v1)
    p1 = rng.integers(0, W, size=(R, W))
    p2 = rng.integers(0, W, size=(R, W))
    h.step(p1)
    h.step(p2)
    k2, _ = h.materialise(2, 3)
    comp = np.take_along_axis(p1, p2, axis=1)          # child b <- p1[p2[b]]
    for r in range(R):
        np.testing.assert_array_equal(k2[r], k0[r][comp[r]])
    with pytest.raises(ValueError):
        h.step(np.full((R, W), W))


# ---------------------------------------------------------------- last valid token
def _last_rows(q_full, cu):
    """The query row of each sequence's last valid token (row 0 for an empty one)."""
    idx = [max(int(cu[i + 1]) - 1, int(cu[i])) for i in range(len(cu) - 1)]
    return np.ascontiguousarray(q_full[np.minimum(idx, max(q_full.shape[0] - 1, 0))])


def test_last_token_equals_last_padded_row():
    """The last-token op is the last row of the causal prefill: checked against the
    independent padded + masked numpy formulation, with an empty sequence in the batch."""
    lengths = [1, 2, 17, 64, 0, 100, 3]
    x = rand_prefill(lengths, 4, 2, 32, seed=61)
    cu = x["cu_seqlens"]
    scale = 1 / math.sqrt(32)
    full = oracle_np.prefill_padded(x["q"], x["k"], x["v"], cu, scale)
    out = oracle.last_token(_last_rows(x["q"], cu), x["k"], x["v"], cu, scale)
    for i, L in enumerate(lengths):
        if L == 0:
            assert np.all(out[i] == 0)               # an empty sequence writes nothing
        else:
            assert np.max(np.abs(out[i] - full[int(cu[i + 1]) - 1])) < 1e-12


def test_last_token_closed_forms():
    # one key: the output is that key's value row, per query head through its kv head
    x = rand_prefill([1, 1], 4, 2, 16, seed=71)
    out = oracle.last_token(x["q"], x["k"], x["v"], x["cu_seqlens"], 0.25)
    kv = widen(x["v"])
    for h in range(4):
        np.testing.assert_array_equal(out[:, h, :], kv[:, h // 2, :])
    # two keys: the logistic weight of the larger logit, and its lse
    fx = json.load(open(os.path.join(GOLDEN, "closed_form_fixtures.json")))["two_keys"]
    d = fx["head_dim"]
    scale = 1.0 / math.sqrt(d)
    q = bits(np.array([[fx["q"]]], dtype=np.float32))
    k = bits(np.array([[fx["k0"]], [fx["k1"]]], dtype=np.float32))
    v = bits(np.array([[fx["v0"]], [fx["v1"]]], dtype=np.float32))
    out, lse = oracle.last_token(q, k, v, np.array([0, 2], np.int32), scale, want_lse=True)
    z0 = scale * (fx["q"][0] * fx["k0"][0] + fx["q"][1] * fx["k0"][1])
    z1 = scale * (fx["q"][0] * fx["k1"][0] + fx["q"][1] * fx["k1"][1])
    w1 = 1.0 / (1.0 + math.exp(z0 - z1))
    for c in range(d):
        assert abs(out[0, 0, c] - ((1 - w1) * fx["v0"][c] + w1 * fx["v1"][c])) < 1e-15
    assert abs(lse[0, 0] - (max(z0, z1) + math.log1p(math.exp(-abs(z0 - z1))))) < 1e-15
    # constant values: every head returns them
    y = rand_prefill([5, 9], 4, 2, 8, seed=81)
    c = np.linspace(-3, 3, 8, dtype=np.float32)
    out = oracle.last_token(_last_rows(y["q"], y["cu_seqlens"]), y["k"], bits(np.broadcast_to(c, y["v"].shape)),
                            y["cu_seqlens"], 1 / math.sqrt(8))
    assert np.max(np.abs(out - widen(bits(c))[None, None, :])) < 1e-14
