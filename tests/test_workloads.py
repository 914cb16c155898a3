"""Seeded input generators: determinism, bf16 rounding and the page's bounds."""
import json
import os

import numpy as np

from attention_packed_varlen_causal_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, -2.5, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, 0.0, -0.0, 3.0e38], np.float32)
    b = wl.bf16_bits_from_f32(f)
    # 1+2^-8 is exactly halfway between 1 and 1+2^-7: ties to even -> 1.0
    assert b.tolist()[:5] == [0x3F80, 0xC020, 0x3F80, 0x3F82, 0x3F80]
    assert b[5] == 0 and b[6] == 0x8000
    assert np.all(wl.bf16_bits_to_f32(b)[[0, 1]] == f[[0, 1]])
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    back = wl.bf16_bits_to_f32(wl.bf16_bits_from_f32(x))
    assert np.max(np.abs(back - x) / np.abs(x)) <= 2**-8


def test_config_sizes_match_recipe():
    assert sum(wl.prefill_lengths(wl.PREFILL_CONFIGS["tiny"])) == 392
    L2 = wl.prefill_lengths(wl.PREFILL_CONFIGS["prefill_only"])
    assert len(L2) == 240 and sum(L2) == 70375 and min(L2) >= 64 and max(L2) <= 500
    L5 = wl.prefill_lengths(wl.PREFILL_CONFIGS["skewed"])
    assert len(L5) == 4096 and sum(L5) == 1356586 and min(L5) >= 1 and max(L5) == 2048
    assert wl.decode_prompt_lengths(wl.DECODE_CONFIGS["beam_long"])[:4] == [485, 464, 451, 427]
    assert wl.decode_prompt_lengths(wl.DECODE_CONFIGS["beam_short"]) == [128] * 32


def test_configs_within_page_bounds():
    b = json.load(open(os.path.join(GOLDEN, "page_bounds.json")))
    L2 = wl.prefill_lengths(wl.PREFILL_CONFIGS["prefill_only"])
    assert np.mean(L2) < b["avg_input_tokens_max"]
    assert len(L2) == 16 * b["prefill_only_samples_per_request"]
    for cfg in wl.DECODE_CONFIGS.values():
        assert cfg.W <= b["beam_width_max"] and cfg.steps <= b["generated_tokens_max"]
        assert np.mean(wl.decode_prompt_lengths(cfg)) < b["avg_input_tokens_max"]
    assert wl.DECODE_CONFIGS["beam_short"].W == b["beam_search_width_reported"]
    assert wl.DECODE_CONFIGS["beam_short"].steps == b["beam_search_decodes_reported"]


def test_generators_deterministic():
    a = wl.make_prefill_inputs([5, 7], 4, 2, 16)
    b = wl.make_prefill_inputs([5, 7], 4, 2, 16)
    for key in ("q", "k", "v", "cu_seqlens"):
        np.testing.assert_array_equal(a[key], b[key])
    c = wl.make_prefill_inputs([5, 7], 4, 2, 16, layer=1)
    assert not np.array_equal(a["k"], c["k"])
    x = wl.make_prefill_inputs([300], 2, 2, 8, outlier_frac=0.01, outlier_scale=8.0)
    y = wl.make_prefill_inputs([300], 2, 2, 8)
    changed = np.any(x["k"] != y["k"], axis=-1)
    assert changed.sum() == 6            # 1% of 600 (token, kv-head) rows
    d = wl.make_decode_problem(2, 3, 2, 4, 2, 8, [4, 0])
    assert d["cu_prompt"].tolist() == [0, 4, 4]
    assert all(p.min() >= 0 and p.max() < 3 for p in d["parent"])


def test_prefix_of_a_configuration_is_the_prefix_of_its_draws():
    # a small per-tensor-seed configuration: the prefix generator must give exactly the
    # first tokens of the whole draw
    cfg = wl.PrefillConfig("small", 7, 4, 2, 64, "uniform", lo=5, hi=40)
    full = wl.make_prefill_config_inputs(cfg, layer=3)
    for n in (1, 3, 7):
        pre = wl.make_prefill_config_prefix(cfg, n, layer=3)
        T = int(full["cu_seqlens"][n])
        assert np.array_equal(pre["cu_seqlens"], full["cu_seqlens"][:n + 1])
        for key in ("q", "k", "v"):
            assert np.array_equal(pre[key], full[key][:T])


def test_prefix_refused_where_it_is_not_a_prefix():
    import pytest
    for name in ("tiny", "skewed"):
        with pytest.raises(ValueError):
            wl.make_prefill_config_prefix(wl.PREFILL_CONFIGS[name], 2)
