"""fp64 CPU oracle for the attention hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never imports, links or executes anything here, and this package
never imports the product.  The only thing both sides share is the seeded
input generator module, which holds no attention arithmetic.

Contents
  * ``prefill(...)``  packed variable-length causal GQA attention, plain fp64
    loops in ``oracle.c`` (abstract + section 1.2 of "SLM 生成式高并发推理引擎：
    延迟约束下的有效吞吐优化": packed prefill computes valid tokens only).
  * ``decode(...)``   attention of each beam's newest query over
    [shared prompt K/V ; the beam's own suffix K/V] (section 1.2: beams of a
    request share one prompt K/V, each keeps a short suffix K/V).
  * ``BeamHistory``   the per-beam suffix as explicit Python lists, advanced
    one decode step at a time by the beam parent index (section 1.1: the
    parent index comes out of beam selection).  The reading used: at step t
    the new history of beam b is the history of beam parent[b] followed by
    beam b's new token (plain reading of sections 1.1 and 1.2).
  * ``oracle_np``     an independent padded-plus-mask numpy formulation used
    to cross-check the C oracle (section 1.2 contrasts padding with packing).
  * ``fp8``           E4M3 codes with one power-of-two scale per tensor, and the
    packed prefill with such Q and K and a bf16 V (the abstract's "selective FP8"; a reading
    for a future FP8 variant of the prefill kernel).  Pins in
    ``tests/test_oracle_fp8_pins.py``.

All pins (closed forms, invariants, brute force) are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "liboracle.so")
# BG_ORACLE_LIB points the oracle at another build of oracle.c; the mutation
# test uses it to load copies with planted mistakes.
_LIB_PATH = os.environ.get("BG_ORACLE_LIB", _DEFAULT_LIB)
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, -O2).

    No -march=native and no intrinsics: the same source builds on x86_64 and
    aarch64 hosts.  -ffp-contract=off keeps every product and sum a separately
    rounded double operation, as written."""
    if _LIB_PATH != _DEFAULT_LIB:
        return _LIB_PATH
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
               "-std=c99", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_prefill.argtypes = [P, P, P, P, i32, i32, i32, i32, ctypes.c_double, P, P]
            lib.oracle_prefill.restype = ctypes.c_int
            lib.oracle_last_token.argtypes = [P, P, P, P, i32, i32, i32, i32, ctypes.c_double, P, P]
            lib.oracle_last_token.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                          ctypes.c_double, P, P]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def prefill(q, k, v, cu_seqlens, scale: float, want_lse: bool = False):
    """Packed causal GQA prefill attention in fp64.

    q: uint16 [T,Hq,d]; k, v: uint16 [T,Hkv,d]; cu_seqlens: int32 [B+1].
    Returns out float64 [T,Hq,d] (and lse float64 [T,Hq] if want_lse)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != (T, Hkv, d) or int(cu[-1]) != T:
        raise ValueError("shape mismatch")
    out = np.zeros((T, Hq, d), dtype=np.float64)
    lse = np.zeros((T, Hq), dtype=np.float64) if want_lse else None
    rc = _load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, Hq, Hkv, d,
                                float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_prefill rejected its arguments (rc={rc})")
    return (out, lse) if want_lse else out


def last_token(q, k, v, cu_seqlens, scale: float, want_lse: bool = False):
    """Attention of each sequence's last valid token over its own keys, in fp64.

    q: uint16 [B,Hq,d] (the last row of each sequence); k, v: uint16 [T,Hkv,d];
    cu_seqlens: int32 [B+1].  Returns float64 [B,Hq,d] (rows of zero-length
    sequences stay 0) and lse float64 [B,Hq] if want_lse."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    B, Hq, d = q.shape
    T, Hkv = k.shape[0], k.shape[1]
    if len(cu) != B + 1 or k.shape != (T, Hkv, d) or v.shape != (T, Hkv, d) or int(cu[-1]) != T:
        raise ValueError("shape mismatch")
    out = np.zeros((B, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64) if want_lse else None
    rc = _load().oracle_last_token(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), B, Hq, Hkv, d, float(scale), _ptr(out),
                                   _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_last_token rejected its arguments (rc={rc})")
    return (out, lse) if want_lse else out


def decode(q, prompt_k, prompt_v, cu_prompt, hist_k, hist_v, scale: float, want_lse: bool = False):
    """Decode attention in fp64 over [prompt_r ; suffix(r,b)].

    q: uint16 [R,W,Hq,d]; prompt_k/v: uint16 [sum P,Hkv,d]; cu_prompt int32
    [R+1]; hist_k/v: uint16 [R,W,t,Hkv,d] (t may be 0).  Returns float64
    [R,W,Hq,d] (and lse [R,W,Hq])."""
    q, pk, pv = _u16(q), _u16(prompt_k), _u16(prompt_v)
    hk, hv = _u16(hist_k), _u16(hist_v)
    cu = np.ascontiguousarray(cu_prompt, dtype=np.int32)
    R, W, Hq, d = q.shape
    Hkv = pk.shape[1]
    t = hk.shape[2]
    if hk.shape != (R, W, t, Hkv, d) or hv.shape != hk.shape or int(cu[-1]) != pk.shape[0]:
        raise ValueError("shape mismatch")
    out = np.zeros((R, W, Hq, d), dtype=np.float64)
    lse = np.zeros((R, W, Hq), dtype=np.float64) if want_lse else None
    rc = _load().oracle_decode(_ptr(q), _ptr(pk), _ptr(pv), _ptr(cu), _ptr(hk), _ptr(hv), t,
                               R, W, Hq, Hkv, d, float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its arguments (rc={rc})")
    return (out, lse) if want_lse else out


class BeamHistory:
    """Per-beam suffix K/V kept as explicit Python lists of rows.

    ``rows[r][b]`` is the list, oldest first, of (k_row, v_row) pairs, each a
    uint16 [Hkv, d] array.  ``step(parent, new_k, new_v)`` implements one
    decode step of the bounded beam search:

        hist'[r][b] = hist[r][parent[r][b]]  followed by  (new_k[r,b], new_v[r,b])

    Several children may share a parent; beams with no child are dropped.
    """

    def __init__(self, R: int, W: int):
        self.R, self.W = R, W
        self.rows: List[List[list]] = [[[] for _ in range(W)] for _ in range(R)]

    def step(self, parent, new_k=None, new_v=None):
        parent = np.asarray(parent)
        if parent.shape != (self.R, self.W):
            raise ValueError("parent shape")
        if parent.min(initial=0) < 0 or parent.max(initial=0) >= self.W:
            raise ValueError("parent index out of range")
        nxt = []
        for r in range(self.R):
            row = []
            for b in range(self.W):
                h = list(self.rows[r][int(parent[r, b])])   # copy the parent's list
                if new_k is not None:
                    h.append((np.array(new_k[r, b], copy=True), np.array(new_v[r, b], copy=True)))
                row.append(h)
            nxt.append(row)
        self.rows = nxt

    def length(self) -> int:
        return len(self.rows[0][0]) if self.R and self.W else 0

    def materialise(self, Hkv: int, d: int):
        """Dense uint16 [R,W,t,Hkv,d] K and V arrays of the current histories."""
        t = self.length()
        hk = np.zeros((self.R, self.W, t, Hkv, d), dtype=np.uint16)
        hv = np.zeros_like(hk)
        for r in range(self.R):
            for b in range(self.W):
                h = self.rows[r][b]
                if len(h) != t:
                    raise ValueError("ragged histories")
                for s, (kr, vr) in enumerate(h):
                    hk[r, b, s] = kr
                    hv[r, b, s] = vr
        return hk, hv
