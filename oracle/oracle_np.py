"""Second, independent fp64 formulation of the oracle -- TEST INFRASTRUCTURE.

Where ``oracle.c`` walks each packed sequence with scalar loops, this module
does the opposite: it *pads* every sequence to the longest one, expands K/V to
all query heads, computes the whole [B, Hq, Lmax, Lmax] score block with one
einsum and removes padded and future keys with a -inf mask.  Section 1.2 of
"SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化" states that packing (valid
tokens only) and padding differ only in wasted work, so both must give the
same numbers.  It is only a cross-check; it is too memory-hungry for the
large workloads.
"""
from __future__ import annotations

import numpy as np


def _widen(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def prefill_padded(q, k, v, cu_seqlens, scale: float) -> np.ndarray:
    """Causal GQA attention via padding + mask.  Returns float64 [T,Hq,d]."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    Q, K, V = _widen(q), _widen(k), _widen(v)
    T, Hq, d = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    B = len(cu) - 1
    lens = cu[1:] - cu[:-1]
    Lmax = int(lens.max()) if B else 0
    Qp = np.zeros((B, Lmax, Hq, d))
    Kp = np.zeros((B, Lmax, Hkv, d))
    Vp = np.zeros((B, Lmax, Hkv, d))
    for i in range(B):
        L = int(lens[i])
        Qp[i, :L] = Q[cu[i]:cu[i + 1]]
        Kp[i, :L] = K[cu[i]:cu[i + 1]]
        Vp[i, :L] = V[cu[i]:cu[i + 1]]
    Kx = np.repeat(Kp, g, axis=2)            # kv-head h//g serves q-head h
    Vx = np.repeat(Vp, g, axis=2)
    s = np.einsum("bphc,bjhc->bhpj", Qp, Kx) * scale
    pos = np.arange(Lmax)
    causal = pos[None, :] <= pos[:, None]                       # [p, j]: j <= p
    valid = pos[None, :] < lens[:, None]                        # [b, j]
    mask = causal[None, None, :, :] & valid[:, None, None, :]
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)                        # padded rows
    w = np.exp(s - m)
    den = w.sum(axis=-1, keepdims=True)
    den = np.where(den > 0, den, 1.0)
    o = np.einsum("bhpj,bjhc->bphc", w / den, Vx)
    out = np.zeros((T, Hq, d))
    for i in range(B):
        L = int(lens[i])
        out[cu[i]:cu[i + 1]] = o[i, :L]
    return out


def full_kv_attention(q, keys, vals, scale: float) -> np.ndarray:
    """Unmasked attention of queries [n, Hq, d] over a materialised key list
    keys/vals [m, Hkv, d] (GQA expanded).  Returns float64 [n, Hq, d]."""
    Q, K, V = _widen(q), _widen(keys), _widen(vals)
    Hq = Q.shape[1]
    g = Hq // K.shape[1]
    Kx = np.repeat(K, g, axis=1)
    Vx = np.repeat(V, g, axis=1)
    s = np.einsum("nhc,jhc->nhj", Q, Kx) * scale
    s = s - s.max(axis=-1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("nhj,jhc->nhc", w, Vx)
