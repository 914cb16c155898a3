"""The work accounting behind every roofline fraction the benchmark reports.

bench.prefill_flops / prefill_bytes / decode_step_work are checked against
quantities counted a different way: query-key pairs counted one by one, bytes
summed tensor by tensor from their shapes, and the per-configuration totals
worked out by hand from the workload definitions (4 FLOPs per multiply-add
pair of QK^T and PV per head dimension; bf16 = 2 bytes).
"""
import numpy as np
import pytest

import bench
from attention_packed_varlen_causal_gb300 import workloads as wl


def _pairs_brute(lengths):
    # causal, self-inclusive: query p of a sequence sees keys 0..p
    return sum(1 for L in lengths for p in range(L) for _ in range(p + 1))


@pytest.mark.parametrize("lengths", [[1], [2, 3], [17, 64, 100, 211], [0, 5, 0, 1]])
def test_prefill_flops_counts_causal_pairs(lengths):
    Hq, d = 16, 128
    # each (query, key, head) pair: d multiply-adds for the logit and d for P.V
    assert bench.prefill_flops(lengths, Hq, d) == 4 * d * Hq * _pairs_brute(lengths)


def test_prefill_bytes_is_q_k_v_read_and_o_written():
    T, Hq, Hkv, d = 392, 16, 8, 128
    q, o = T * Hq * d * 2, T * Hq * d * 2
    k = v = T * Hkv * d * 2
    assert bench.prefill_bytes(T, Hq, Hkv, d) == q + k + v + o


@pytest.mark.parametrize("name,gflop,mb", [
    ("tiny", 0.243, 4.8),            # 4 sequences {17, 64, 100, 211}
    ("prefill_only", 101.6, 864.8),  # 240 sequences, T = 70,375
    ("skewed", 3331.6, 16669.7),     # 4096 sequences, T = 1,356,586
])
def test_prefill_config_totals(name, gflop, mb):
    cfg = wl.PREFILL_CONFIGS[name]
    L = wl.prefill_lengths(cfg)
    T = int(wl.cu_from_lengths(L)[-1])
    assert bench.prefill_flops(L, cfg.Hq, cfg.head_dim) / 1e9 == pytest.approx(gflop, rel=2e-3)
    assert bench.prefill_bytes(T, cfg.Hq, cfg.Hkv, cfg.head_dim) / 1e6 == pytest.approx(mb, abs=0.1)


def _decode_bytes_by_tensor(cfg, plen, t):
    R, W, Hq, Hkv, d = cfg.R, cfg.W, cfg.Hq, cfg.Hkv, cfg.head_dim
    b2 = 2                                               # bf16
    q = R * W * Hq * d * b2                              # the step's queries, read once
    o = R * W * Hq * d * b2                              # the output, written once
    prompt = 2 * sum(plen) * Hkv * d * b2                # prompt K and V, read once per request
    slot_kv = 2 * R * W * Hkv * d * b2                   # one suffix slot of K and V over all beams
    reorder = (t - 1) * slot_kv * 2                      # slots 0..t-2 read from the parents, written
    append = slot_kv * 2                                 # the new token's K/V read, written to slot t-1
    suffix_read = t * slot_kv                            # the attention reads slots 0..t-1
    return q + o + prompt + reorder + append + suffix_read


@pytest.mark.parametrize("name", ["beam_short", "beam_long"])
@pytest.mark.parametrize("t", [1, 2, 5])
def test_decode_step_work_by_tensor(name, t):
    cfg = wl.DECODE_CONFIGS[name]
    plen = wl.decode_prompt_lengths(cfg)
    flops, by = bench.decode_step_work(cfg, plen, t)
    # every (request, beam, q head) row attends over its request's prompt and t suffix keys
    rows_keys = sum(cfg.W * cfg.Hq * (P + t) for P in plen)
    assert flops == pytest.approx(4 * cfg.head_dim * rows_keys, rel=1e-12)
    assert by == pytest.approx(_decode_bytes_by_tensor(cfg, plen, t), rel=1e-12)


def test_decode_prompt_phase_matches_worked_figures():
    # short prompt: 32 x 128-token prompts, beam 100, 14 q heads, d 64 -> 1.47 GFLOP;
    # Q 5.7 MB + O 5.7 MB + prompt K/V 2.1 MB per step
    cfg = wl.DECODE_CONFIGS["beam_short"]
    plen = wl.decode_prompt_lengths(cfg)
    f1, _ = bench.decode_step_work(cfg, plen, 1)
    suffix_flops = 4 * cfg.head_dim * cfg.R * cfg.W * cfg.Hq * 1
    assert (f1 - suffix_flops) / 1e9 == pytest.approx(1.468, abs=0.001)
    prompt_phase = _decode_bytes_by_tensor(cfg, plen, 1) - 2 * (2 * cfg.R * cfg.W * cfg.Hkv * cfg.head_dim * 2) \
        - (2 * cfg.R * cfg.W * cfg.Hkv * cfg.head_dim * 2)
    assert prompt_phase / 1e6 == pytest.approx(13.57, abs=0.01)
    # long prompt: 16 prompts of 7,208 tokens in all, beam 400 -> 10.33 GFLOP
    cfg = wl.DECODE_CONFIGS["beam_long"]
    plen = wl.decode_prompt_lengths(cfg)
    assert sum(plen) == 7208
    f1, _ = bench.decode_step_work(cfg, plen, 1)
    suffix_flops = 4 * cfg.head_dim * cfg.R * cfg.W * cfg.Hq * 1
    assert (f1 - suffix_flops) / 1e9 == pytest.approx(10.33, abs=0.005)


def test_first_step_moves_no_parent_slots():
    # t = 1: nothing to reorder; the step's bytes exceed step 1's attention reads only by the append
    cfg = wl.DECODE_CONFIGS["beam_short"]
    plen = wl.decode_prompt_lengths(cfg)
    _, b1 = bench.decode_step_work(cfg, plen, 1)
    _, b2 = bench.decode_step_work(cfg, plen, 2)
    slot_kv = 2 * cfg.R * cfg.W * cfg.Hkv * cfg.head_dim * 2
    # one more slot reordered (read + write) and one more suffix slot read by the attention
    assert b2 - b1 == pytest.approx(3 * slot_kv, rel=1e-12)
    assert np.isfinite(b1)


def test_decode_item_spread():
    # 18-beam query tiles (g = 7), two per item, round-robin over 152 CTAs
    short = wl.DECODE_CONFIGS["beam_short"]       # 100 beams: 6 tiles -> 3 items per (request, kv head)
    assert bench.decode_item_spread(short, 152) == (32 * 2 * 3, 152, 2)
    long_ = wl.DECODE_CONFIGS["beam_long"]        # 400 beams: 23 tiles -> 12 items per (request, kv head)
    assert bench.decode_item_spread(long_, 152) == (16 * 2 * 12, 152, 3)
    assert bench.decode_item_spread(short, 1000) == (192, 192, 1)
