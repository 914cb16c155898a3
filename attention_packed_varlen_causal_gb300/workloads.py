"""Seeded synthetic inputs for the attention hot path.

This module only *draws inputs*: sequence lengths, bf16 Q/K/V bit patterns,
beam parent indices.  It holds none of the attention arithmetic, so both the
CUDA path (through the binding) and the CPU oracle can be fed from it without
sharing any of the method's code.

Workload shapes follow the bounded-generation SLM engine described in
"SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化" (163.com), section 1.2
(input/state bounds): average inputs under 500 tokens, Prefill-Only requests
carrying several samples, beam width at most 400 and at most 5 generated
tokens.  The exact sizes (head counts, head dim, GQA ratio) are the five
configurations below; the pages themselves fix none of them.

bf16 values are produced by drawing fp32 N(0,1) with numpy's PCG64
``default_rng`` and rounding to bf16 with round-to-nearest-even; the *same*
uint16 bit patterns go to the GPU and to the oracle.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "bf16_bits_from_f32", "bf16_bits_to_f32", "PrefillConfig", "DecodeConfig",
    "PREFILL_CONFIGS", "DECODE_CONFIGS", "prefill_lengths", "make_prefill_inputs",
    "make_decode_problem", "cu_from_lengths",
]


# ---------------------------------------------------------------------------
# bf16 bit handling (input preparation, not attention arithmetic)
# ---------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even) and return the raw
    uint16 bit patterns.  NaN is not produced by the generators."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding_bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding_bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(size=shape, dtype=np.float32))


# ---------------------------------------------------------------------------
# Configurations
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    head_dim: int
    length_kind: str            # "fixed" | "uniform" | "lognormal"
    fixed_lengths: tuple = ()
    lo: int = 0
    hi: int = 0
    mu: float = 0.0
    sigma: float = 0.0
    outlier_frac: float = 0.0   # fraction of (token, kv-head) K rows scaled
    outlier_scale: float = 1.0
    single_seed_qkv: Optional[int] = None   # draw q,k,v in order from one rng
    layers: int = 1


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    R: int                      # requests
    W: int                      # beam width
    steps: int                  # decode steps (suffix length 1..steps)
    Hq: int
    Hkv: int
    head_dim: int
    prompt_fixed: int = 0       # >0: every request has this prompt length
    prompt_lo: int = 0
    prompt_hi: int = 0
    layers: int = 1


PREFILL_CONFIGS: Dict[str, PrefillConfig] = {
    # 4 sequences {17, 64, 100, 211}, GQA 16/8, d 128, q/k/v from one seed-0 rng
    "tiny": PrefillConfig("tiny", 4, 16, 8, 128, "fixed", fixed_lengths=(17, 64, 100, 211),
                          single_seed_qkv=0),
    # Prefill-Only request batch: 16 requests x 15 samples, L ~ U{64..500}
    "prefill_only": PrefillConfig("prefill_only", 240, 16, 8, 128, "uniform", lo=64, hi=500,
                                  layers=28),
    # skewed stress: 4096 sequences, L = clip(round(lognormal(5.5, 0.8)), 1, 2048),
    # 1% of K rows scaled x8 (outlier logits)
    "skewed": PrefillConfig("skewed", 4096, 16, 8, 128, "lognormal", lo=1, hi=2048, mu=5.5,
                            sigma=0.8, outlier_frac=0.01, outlier_scale=8.0),
}

DECODE_CONFIGS: Dict[str, DecodeConfig] = {
    # short prompt: 32 requests x 128-token prompt, beam 100, 4 steps, 14/2 heads, d 64
    "beam_short": DecodeConfig("beam_short", 32, 100, 4, 14, 2, 64, prompt_fixed=128, layers=28),
    # long prompt: 16 requests, prompt ~ U{400..500}, beam 400, 5 steps
    "beam_long": DecodeConfig("beam_long", 16, 400, 5, 14, 2, 64, prompt_lo=400, prompt_hi=500,
                              layers=28),
}

# seeds: lengths 0; Q/K/V 1/2/3 (+100*layer); new-token K/V 4 (+100*layer);
# parent_idx 5 + step (+100*layer is not applied: parents are per model step);
# K outlier rows 6; decode queries 7 (+100*layer, +1000*step)
SEED_LEN, SEED_Q, SEED_K, SEED_V, SEED_NEWKV, SEED_PARENT, SEED_OUTLIER, SEED_DQ = 0, 1, 2, 3, 4, 5, 6, 7


def prefill_lengths(cfg: PrefillConfig) -> List[int]:
    if cfg.length_kind == "fixed":
        return list(cfg.fixed_lengths)
    rng = np.random.default_rng(SEED_LEN)
    if cfg.length_kind == "uniform":
        return rng.integers(cfg.lo, cfg.hi + 1, size=cfg.num_seqs).astype(int).tolist()
    if cfg.length_kind == "lognormal":
        x = np.round(rng.lognormal(cfg.mu, cfg.sigma, size=cfg.num_seqs))
        return np.clip(x, cfg.lo, cfg.hi).astype(int).tolist()
    raise ValueError(cfg.length_kind)


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if cu[-1] >= 2**31:
        raise ValueError("total tokens exceed int32")
    return cu.astype(np.int32)


def make_prefill_inputs(lengths, Hq: int, Hkv: int, head_dim: int, *, layer: int = 0,
                        single_seed: Optional[int] = None, outlier_frac: float = 0.0,
                        outlier_scale: float = 1.0, seeds=None) -> dict:
    """Packed Q [T,Hq,d], K/V [T,Hkv,d] as bf16 bits (uint16), cu_seqlens int32 [B+1].

    ``seeds`` optionally overrides (q, k, v) seeds, e.g. for tests that need
    several independent draws."""
    cu = cu_from_lengths(lengths)
    T = int(cu[-1])
    if single_seed is not None:
        rng = np.random.default_rng(single_seed)
        q = _normal_bf16(rng, (T, Hq, head_dim))
        k = _normal_bf16(rng, (T, Hkv, head_dim))
        v = _normal_bf16(rng, (T, Hkv, head_dim))
    else:
        sq, sk, sv = seeds if seeds is not None else (SEED_Q, SEED_K, SEED_V)
        off = 100 * layer
        q = _normal_bf16(np.random.default_rng(sq + off), (T, Hq, head_dim))
        k_f = np.random.default_rng(sk + off).standard_normal(size=(T, Hkv, head_dim), dtype=np.float32)
        if outlier_frac > 0.0:
            rows = T * Hkv
            n_out = int(round(outlier_frac * rows))
            pick = np.random.default_rng(SEED_OUTLIER + off).choice(rows, size=n_out, replace=False)
            k_f.reshape(rows, head_dim)[pick] *= np.float32(outlier_scale)
        k = bf16_bits_from_f32(k_f)
        v = _normal_bf16(np.random.default_rng(sv + off), (T, Hkv, head_dim))
    return {"q": q, "k": k, "v": v, "cu_seqlens": cu, "lengths": list(lengths),
            "Hq": Hq, "Hkv": Hkv, "head_dim": head_dim, "max_seqlen": int(max(lengths) if len(lengths) else 0)}


def make_prefill_config_prefix(cfg: PrefillConfig, n_seqs: int, layer: int = 0) -> dict:
    """The first ``n_seqs`` sequences of a configuration's inputs, without drawing the rest.

    With one generator per tensor, the first n values a generator draws do not depend on
    how many it draws in all, so the first T' tokens of Q, K and V come out exactly as in
    the whole configuration.  That holds only without a shared generator and without
    outlier rows (their choice depends on T); other configurations are refused."""
    if cfg.single_seed_qkv is not None or cfg.outlier_frac > 0.0:
        raise ValueError(f"{cfg.name}: a prefix of its inputs is not a prefix of the draws")
    lengths = prefill_lengths(cfg)[:n_seqs]
    return make_prefill_inputs(lengths, cfg.Hq, cfg.Hkv, cfg.head_dim, layer=layer)


def make_prefill_config_inputs(cfg: PrefillConfig, layer: int = 0) -> dict:
    return make_prefill_inputs(prefill_lengths(cfg), cfg.Hq, cfg.Hkv, cfg.head_dim, layer=layer,
                               single_seed=cfg.single_seed_qkv, outlier_frac=cfg.outlier_frac,
                               outlier_scale=cfg.outlier_scale)


def decode_prompt_lengths(cfg: DecodeConfig) -> List[int]:
    if cfg.prompt_fixed > 0:
        return [cfg.prompt_fixed] * cfg.R
    rng = np.random.default_rng(SEED_LEN)
    return rng.integers(cfg.prompt_lo, cfg.prompt_hi + 1, size=cfg.R).astype(int).tolist()


def make_decode_problem(R: int, W: int, steps: int, Hq: int, Hkv: int, head_dim: int,
                        prompt_lengths, *, layer: int = 0) -> dict:
    """Everything one beam-search decode of ``steps`` steps consumes, per layer:

    prompt K/V packed [sum P, Hkv, d] + cu_prompt [R+1]; per step s (0-based):
    query q[s] [R,W,Hq,d], the new token's K/V new_k[s]/new_v[s] [R,W,Hkv,d],
    parent[s] [R,W] int32 in [0,W).  The parent of step 0 is drawn too (it
    moves zero suffix tokens)."""
    cu = cu_from_lengths(prompt_lengths)
    Ptot = int(cu[-1])
    off = 100 * layer
    pk = _normal_bf16(np.random.default_rng(SEED_K + off), (Ptot, Hkv, head_dim))
    pv = _normal_bf16(np.random.default_rng(SEED_V + off), (Ptot, Hkv, head_dim))
    qs, nks, nvs, parents = [], [], [], []
    for s in range(steps):
        qs.append(_normal_bf16(np.random.default_rng(SEED_DQ + off + 1000 * s), (R, W, Hq, head_dim)))
        rng_kv = np.random.default_rng(SEED_NEWKV + off + 1000 * s)
        nks.append(_normal_bf16(rng_kv, (R, W, Hkv, head_dim)))
        nvs.append(_normal_bf16(rng_kv, (R, W, Hkv, head_dim)))
        parents.append(np.random.default_rng(SEED_PARENT + s).integers(0, W, size=(R, W)).astype(np.int32))
    return {"prompt_k": pk, "prompt_v": pv, "cu_prompt": cu, "prompt_lengths": list(prompt_lengths),
            "q": qs, "new_k": nks, "new_v": nvs, "parent": parents, "R": R, "W": W, "steps": steps,
            "Hq": Hq, "Hkv": Hkv, "head_dim": head_dim,
            "max_prompt_len": int(max(prompt_lengths) if len(prompt_lengths) else 0)}


def make_decode_config_problem(cfg: DecodeConfig, layer: int = 0) -> dict:
    return make_decode_problem(cfg.R, cfg.W, cfg.steps, cfg.Hq, cfg.Hkv, cfg.head_dim,
                               decode_prompt_lengths(cfg), layer=layer)
