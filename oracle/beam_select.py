"""Beam candidate selection, plain fp64 numpy -- TEST INFRASTRUCTURE.

Same rules as the rest of ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may use it; it never imports the product.

Page: "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.1: after the
prompt prefill a beam-search request runs a fixed number of decode steps; the
first step's logits initialise the candidates, and every later step selects
local candidates from each beam's token distribution, merges them with the
accumulated scores and keeps a fixed number W of candidate sequences.  The
candidates, the accumulated scores and the parent index come out of it.

Readings (the page gives no formula):
  * the token distribution of beam b is the softmax over the vocabulary of its
    next-token logits; scores are log-probabilities and accumulate by addition:
        score(b, v) = cum[b] + logits[b, v] - logsumexp_u(logits[b, u]);
  * the W kept candidates are the W largest scores over all (b, v); the local
    candidates of a beam are its own W best tokens, which contain that beam's
    whole share of the global W best, so selecting per beam and then merging
    equals the global selection written here;
  * the kept candidates are ordered by score, highest first, and equal scores
    by the smaller flat index b * V + v;
  * the first step is the same selection with only beam 0 alive
    (cum = [0, -inf, ..., -inf]);
  * outputs per kept candidate: its token v, its parent beam b, its score.
"""
from __future__ import annotations

import numpy as np


def log_softmax_rows(logits) -> np.ndarray:
    """log softmax over the last axis, in fp64 (max subtracted first)."""
    x = np.asarray(logits, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    return x - (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))


def beam_select(logits, cum):
    """logits [R, W, V] (any float type; widened exactly to fp64), cum [R, W].

    Returns (token [R, W] int32, parent [R, W] int32, score [R, W] float64): the
    W best candidates of every request in the order stated above."""
    x = np.asarray(logits, dtype=np.float64)
    if x.ndim != 3:
        raise ValueError("logits must be [R, W, V]")
    R, W, V = x.shape
    c = np.asarray(cum, dtype=np.float64).reshape(R, W)
    lp = log_softmax_rows(x)
    token = np.empty((R, W), dtype=np.int32)
    parent = np.empty((R, W), dtype=np.int32)
    score = np.empty((R, W), dtype=np.float64)
    flat_index = np.arange(W * V, dtype=np.int64)
    for r in range(R):
        s = (c[r][:, None] + lp[r]).reshape(-1)            # candidate (b, v) at b * V + v
        order = np.lexsort((flat_index, -s))                # score descending, then flat index
        keep = order[:W]
        parent[r] = (keep // V).astype(np.int32)
        token[r] = (keep % V).astype(np.int32)
        score[r] = s[keep]
    return token, parent, score
