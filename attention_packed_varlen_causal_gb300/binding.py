"""Thin ctypes binding over ``libbgattn.so`` (the C ABI in include/bg_attn.h).

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream straight to the library; all of the work runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
or fails to load, every call raises.

The functions carry the C names.  Tensor arguments are torch CUDA tensors
(torch is used for device memory and streams only); ``raw`` exposes the
ctypes functions themselves for callers that manage pointers directly.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbgattn.so")

BG_OK, BG_ERR_INVALID_ARG, BG_ERR_UNSUPPORTED, BG_ERR_DEVICE_DATA, BG_ERR_CUDA = 0, 1, 2, 3, 4
BG_DEVSTAT_CU_SEQLENS = 0x01
BG_DEVSTAT_SEQ_TOO_LONG = 0x02
BG_DEVSTAT_PARENT = 0x04
BG_DEVSTAT_CU_PROMPT = 0x08
BG_DEVSTAT_EMPTY_ROW = 0x10
BG_DEVSTAT_PLAN = 0x20
BG_DEVSTAT_TIMEOUT = 0x100
BG_MAX_SUFFIX = 16
BG_MAX_SEQLEN = 65536
BG_NOALLOC_SCRATCH_BYTES = 1 << 20
BG_MAX_BEAM = 512
BG_MAX_VOCAB = 1 << 22

# Every symbol include/bg_attn.h declares, with its ctypes signature.
_P, _I32, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "bg_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "bg_packed_prefill_workspace_size": ([_I32] * 6, _SZ),
    "bg_packed_prefill_attn": ([_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P, _SZ, _P, _P],
                               ctypes.c_int),
    "bg_packed_prefill_plan": ([_P, _I32, _I32, _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "bg_packed_prefill_attn_planned": ([_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P, _SZ, _P,
                                        _P], ctypes.c_int),
    "bg_packed_prefill_attn_fp8": ([_P, _F32, _P, _F32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P,
                                    _SZ, _P, _P], ctypes.c_int),
    "bg_packed_prefill_attn_noalloc": ([_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P, _P],
                                       ctypes.c_int),
    "bg_packed_last_token_attn": ([_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _P, _P, _P],
                                  ctypes.c_int),
    "bg_beam_decode_attn": ([_P, _P, _P, _P, _I32, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P,
                             _P, _P], ctypes.c_int),
    "bg_beam_suffix_reorder": ([_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P],
                               ctypes.c_int),
    "bg_beam_decode_step": ([_P, _P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                             _I32, _I32, _F32, _P, _P, _P], ctypes.c_int),
    "bg_beam_select_workspace_size": ([_I32] * 3, _SZ),
    "bg_selftest_wait_timeout": ([_P, _P, _P], ctypes.c_int),
    "bg_beam_select": ([_P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
}


class BgError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


_lib = None


def load(path: Optional[str] = None):
    """Load the library (once).  Raises if it is not built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with attention_packed_varlen_causal_gb300.build.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


class _Raw:
    def __getattr__(self, name):
        return getattr(load(), name)


raw = _Raw()


def status_string(status: int) -> str:
    return load().bg_status_string(int(status)).decode()


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(fn: str, status: int):
    if status != BG_OK:
        raise BgError(fn, status)


def bg_packed_prefill_workspace_size(num_seqs: int, total_tokens: int, max_seqlen: int, Hq: int, Hkv: int,
                                     head_dim: int) -> int:
    return int(load().bg_packed_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, Hq, Hkv, head_dim))


def bg_packed_prefill_attn(q, k, v, cu_seqlens, max_seqlen: int, out, *, lse=None, scale: Optional[float] = None,
                           workspace=None, dev_status=None, stream=None):
    """q [T,Hq,d], k/v [T,Hkv,d] bf16 CUDA tensors; cu_seqlens int32 [B+1] CUDA;
    out bf16 [T,Hq,d] (written); lse fp32 [T,Hq] or None; workspace a uint8
    CUDA tensor of at least bg_packed_prefill_workspace_size bytes."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bg_packed_prefill_workspace_size(B, T, max_seqlen, Hq, Hkv, d)
    if workspace is None:
        raise ValueError(f"workspace of {need} bytes required (the library never allocates)")
    st = load().bg_packed_prefill_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, T, int(max_seqlen), Hq, Hkv, d,
                                       float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                       _stream(stream))
    _check("bg_packed_prefill_attn", st)
    return out


def bg_packed_prefill_plan(cu_seqlens, total_tokens: int, max_seqlen: int, *, workspace=None, dev_status=None,
                           stream=None):
    """The work list of a packing (cu_seqlens int32 [B+1] CUDA) into workspace, for
    bg_packed_prefill_attn_planned calls with the same packing."""
    B = cu_seqlens.numel() - 1
    if workspace is None:
        raise ValueError("workspace required (the library never allocates)")
    st = load().bg_packed_prefill_plan(_ptr(cu_seqlens), B, int(total_tokens), int(max_seqlen), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                       _stream(stream))
    _check("bg_packed_prefill_plan", st)


def bg_packed_prefill_attn_planned(q, k, v, cu_seqlens, max_seqlen: int, out, *, lse=None,
                                   scale: Optional[float] = None, workspace=None, dev_status=None, stream=None):
    """bg_packed_prefill_attn with the work list a bg_packed_prefill_plan call left in
    workspace (same cu_seqlens, max_seqlen and total tokens)."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        raise ValueError("workspace required (the library never allocates)")
    st = load().bg_packed_prefill_attn_planned(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, T, int(max_seqlen), Hq,
                                               Hkv, d, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                               workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                               _stream(stream))
    _check("bg_packed_prefill_attn_planned", st)
    return out


def bg_packed_prefill_attn_fp8(q_codes, q_scale: float, k_codes, k_scale: float, v, cu_seqlens, max_seqlen: int, out,
                               *, lse=None, scale: Optional[float] = None, workspace=None, dev_status=None,
                               stream=None):
    """q_codes uint8 [T,Hq,d] and k_codes uint8 [T,Hkv,d] E4M3 codes (torch.uint8 or
    torch.float8_e4m3fn CUDA tensors) with their per-tensor scales; v bf16 [T,Hkv,d];
    cu_seqlens int32 [B+1]; out bf16 [T,Hq,d] (written); lse fp32 [T,Hq] or None; workspace
    as for bg_packed_prefill_attn.  ``scale`` is the softmax scale of the dequantised
    values (default 1/sqrt(d))."""
    T, Hq, d = q_codes.shape
    Hkv = k_codes.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bg_packed_prefill_workspace_size(B, T, max_seqlen, Hq, Hkv, d)
    if workspace is None:
        raise ValueError(f"workspace of {need} bytes required (the library never allocates)")
    st = load().bg_packed_prefill_attn_fp8(_ptr(q_codes), float(q_scale), _ptr(k_codes), float(k_scale), _ptr(v),
                                           _ptr(cu_seqlens), B, T, int(max_seqlen), Hq, Hkv, d, float(scale), _ptr(out),
                                           _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _ptr(dev_status), _stream(stream))
    _check("bg_packed_prefill_attn_fp8", st)
    return out


def bg_packed_prefill_attn_noalloc(q, k, v, cu_seqlens, max_seqlen: int, out, *, lse=None,
                                   scale: Optional[float] = None, dev_status=None, stream=None):
    """As bg_packed_prefill_attn, for callers that cannot allocate: the work
    list lives in the library's own fixed device array (no workspace
    argument).  Calls on one device share that array, so calls that can
    overlap on the GPU must be serialised; the first call on a device should
    precede any stream capture."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = load().bg_packed_prefill_attn_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, T, int(max_seqlen), Hq,
                                               Hkv, d, float(scale), _ptr(out), _ptr(lse), _ptr(dev_status),
                                               _stream(stream))
    _check("bg_packed_prefill_attn_noalloc", st)
    return out


def bg_packed_last_token_attn(q, k, v, cu_seqlens, max_seqlen: int, out, *, lse=None,
                              scale: Optional[float] = None, dev_status=None, stream=None):
    """q [B,Hq,d] (each sequence's last valid row); k, v [T,Hkv,d]; cu_seqlens
    int32 [B+1]; out [B,Hq,d] (written); lse fp32 [B,Hq] or None."""
    B, Hq, d = q.shape
    T, Hkv = k.shape[0], k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = load().bg_packed_last_token_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, T, int(max_seqlen), Hq,
                                          Hkv, d, float(scale), _ptr(out), _ptr(lse), _ptr(dev_status),
                                          _stream(stream))
    _check("bg_packed_last_token_attn", st)
    return out


def bg_beam_decode_attn(q, prompt_k, prompt_v, cu_prompt, max_prompt_len: int, suffix_k, suffix_v, suffix_len: int,
                        out, *, scale: Optional[float] = None, dev_status=None, stream=None):
    """q [R,W,Hq,d]; prompt_k/v [sumP,Hkv,d]; cu_prompt int32 [R+1];
    suffix_k/v [R,W,S_max,Hkv,d]; out [R,W,Hq,d] (written)."""
    R, W, Hq, d = q.shape
    Hkv = prompt_k.shape[1]
    S_max = suffix_k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = load().bg_beam_decode_attn(_ptr(q), _ptr(prompt_k), _ptr(prompt_v), _ptr(cu_prompt), prompt_k.shape[0],
                                    int(max_prompt_len), _ptr(suffix_k), _ptr(suffix_v), int(suffix_len), S_max, R, W,
                                    Hq, Hkv, d, float(scale), _ptr(out), _ptr(dev_status), _stream(stream))
    _check("bg_beam_decode_attn", st)
    return out


def bg_beam_suffix_reorder(src_k, src_v, dst_k, dst_v, parent_idx, n_tokens: int, *, new_k=None, new_v=None,
                           dev_status=None, stream=None):
    """src/dst [R,W,S_max,Hkv,d] bf16; parent_idx int32 [R,W]; new_k/new_v
    [R,W,Hkv,d] or None.  dst[r,b,:n] = src[r,parent[r,b],:n], dst[r,b,n] = new[r,b]."""
    R, W, S_max, Hkv, d = src_k.shape
    st = load().bg_beam_suffix_reorder(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v), _ptr(parent_idx),
                                       _ptr(new_k), _ptr(new_v), R, W, S_max, int(n_tokens), Hkv, d,
                                       _ptr(dev_status), _stream(stream))
    _check("bg_beam_suffix_reorder", st)
    return dst_k, dst_v


def bg_beam_decode_step(q, prompt_k, prompt_v, cu_prompt, max_prompt_len: int, src_suffix_k, src_suffix_v,
                        parent_idx, new_k, new_v, dst_suffix_k, dst_suffix_v, suffix_len: int, out, *,
                        scale: Optional[float] = None, dev_status=None, stream=None):
    """One decode step in one call: dst[r,b,:t-1] = src[r,parent[r,b],:t-1], dst[r,b,t-1] = new[r,b],
    then out = decode attention over [prompt ; dst[:, :, :t]] (t = suffix_len >= 1).
    src/dst [R,W,S_max,Hkv,d] bf16 (src may be None when t == 1); parent_idx int32 [R,W];
    new_k/new_v [R,W,Hkv,d]; out [R,W,Hq,d] (written)."""
    R, W, Hq, d = q.shape
    Hkv = prompt_k.shape[1]
    S_max = dst_suffix_k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = load().bg_beam_decode_step(_ptr(q), _ptr(prompt_k), _ptr(prompt_v), _ptr(cu_prompt), prompt_k.shape[0],
                                    int(max_prompt_len), _ptr(src_suffix_k), _ptr(src_suffix_v), _ptr(parent_idx),
                                    _ptr(new_k), _ptr(new_v), _ptr(dst_suffix_k), _ptr(dst_suffix_v),
                                    int(suffix_len), S_max, R, W, Hq, Hkv, d, float(scale), _ptr(out),
                                    _ptr(dev_status), _stream(stream))
    _check("bg_beam_decode_step", st)
    return out


def bg_selftest_wait_timeout(dev_status, waited_ns, *, stream=None):
    """Makes one bounded pipeline wait run out on the device: dev_status (int32) receives
    BG_DEVSTAT_TIMEOUT, waited_ns (int64) the nanoseconds waited."""
    st = load().bg_selftest_wait_timeout(_ptr(dev_status), _ptr(waited_ns), _stream(stream))
    _check("bg_selftest_wait_timeout", st)


def bg_beam_select_workspace_size(R: int, W: int, V: int) -> int:
    return int(load().bg_beam_select_workspace_size(R, W, V))


def bg_beam_select(logits, cum, token_out, parent_out, score_out, *, workspace=None, stream=None):
    """logits fp32 [R,W,V]; cum fp32 [R,W]; token_out/parent_out int32 [R,W] and
    score_out fp32 [R,W] (written); workspace a uint8 CUDA tensor of at least
    bg_beam_select_workspace_size bytes."""
    R, W, V = logits.shape
    need = bg_beam_select_workspace_size(R, W, V)
    if workspace is None:
        raise ValueError(f"workspace of {need} bytes required (the library never allocates)")
    st = load().bg_beam_select(_ptr(logits), _ptr(cum), R, W, V, _ptr(token_out), _ptr(parent_out), _ptr(score_out),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("bg_beam_select", st)
    return token_out, parent_out, score_out
