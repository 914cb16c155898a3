"""GPU check of the prefill -> decode handoff of a beam-search request.

Page 1, "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化", section 1.2: the beams of a
request share the one prompt K/V that its prefill produced, and each beam keeps its own
short suffix K/V; section 1.1: a beam search is one prefill plus a fixed number of decode
steps whose parent index reorders the suffix.  Here the K/V that bg_packed_prefill_attn
reads (packed by cu_seqlens) is handed, in the same device buffers and with cu_seqlens as
cu_prompt, to bg_beam_decode_step for several steps:
  * the prefill output and every step's decode output match the fp64 oracle;
  * the suffix left in dst equals the oracle's explicit per-beam histories bit for bit;
  * the decode output of every (request, beam) equals the last row of a GPU prefill over
    the sequence prompt_r ++ history(b) whose last query is that beam's query (the
    oracle's cross-mode equivalence, run on the GPU), within the parity tolerance."""
import math

import numpy as np
import pytest

import oracle
from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from attention_packed_varlen_causal_gb300 import workloads as wl
from tests.helpers import assert_parity, bits_from_dev, from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


def _prefill(q, k, v, cu, max_len):
    """bg_packed_prefill_attn on device tensors; returns the output tensor."""
    import torch
    T, Hq, d = q.shape
    out = torch.full((T, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bg.bg_packed_prefill_workspace_size(cu.numel() - 1, T, max_len, Hq, k.shape[1], d),
                     dtype=torch.uint8, device="cuda")
    bg.bg_packed_prefill_attn(q, k, v, cu, max_len, out, workspace=ws)
    return out


@pytest.mark.parametrize("Hq,Hkv,d,W,prompts,steps", [
    (14, 2, 64, 5, [37, 130, 64], 3),
    (16, 8, 128, 4, [200, 1, 129], 3),
])
def test_prefill_kv_feeds_decode_unchanged(Hq, Hkv, d, W, prompts, steps):
    import torch
    R = len(prompts)
    scale = 1.0 / math.sqrt(d)
    # the request batch's prefill: prompt tokens packed by cu_seqlens
    px = wl.make_prefill_inputs(prompts, Hq, Hkv, d, seeds=(301, 302, 303))
    cu_np = px["cu_seqlens"]
    q_pre, k_pre, v_pre = to_dev(px["q"]), to_dev(px["k"]), to_dev(px["v"])
    cu = i32_dev(cu_np)
    out_pre = _prefill(q_pre, k_pre, v_pre, cu, max(prompts))
    torch.cuda.synchronize()
    want_pre = oracle.prefill(px["q"], px["k"], px["v"], cu_np, scale)
    assert_parity(from_dev(out_pre), want_pre, "prefill of the prompts")

    # the decode steps take the prefill's K/V buffers and cu_seqlens as they are
    pr = wl.make_decode_problem(R, W, steps, Hq, Hkv, d, prompts, layer=7)
    k_snapshot = bits_from_dev(k_pre).copy()
    hist = oracle.BeamHistory(R, W)
    sk = [torch.full((R, W, steps, Hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    sv = [torch.full((R, W, steps, Hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for s in range(steps):
        src, dst = s % 2, 1 - s % 2
        q = to_dev(pr["q"][s])
        out = torch.empty_like(q)
        bg.bg_beam_decode_step(q, k_pre, v_pre, cu, max(prompts), sk[src] if s else None, sv[src] if s else None,
                               i32_dev(pr["parent"][s]), to_dev(pr["new_k"][s]), to_dev(pr["new_v"][s]), sk[dst],
                               sv[dst], s + 1, out)
        torch.cuda.synchronize()
        hist.step(pr["parent"][s], pr["new_k"][s], pr["new_v"][s])
        hk, hv = hist.materialise(Hkv, d)
        assert np.array_equal(bits_from_dev(sk[dst])[:, :, :s + 1], hk), f"step {s + 1}: suffix K"
        assert np.array_equal(bits_from_dev(sv[dst])[:, :, :s + 1], hv), f"step {s + 1}: suffix V"
        got = from_dev(out)
        want = oracle.decode(pr["q"][s], px["k"], px["v"], cu_np, hk, hv, scale)
        assert_parity(got, want, f"decode step {s + 1} vs oracle")

        # the same rows from the prefill kernel: one sequence per (r, b), prompt_r ++ history(b),
        # whose last query row is the beam's decode query
        seq_q, seq_k, seq_v, lens = [], [], [], []
        for r in range(R):
            a, e = int(cu_np[r]), int(cu_np[r + 1])
            for b in range(W):
                # the history positions' own queries do not matter here: the beam's query fills them
                seq_q.append(np.concatenate([px["q"][a:e], np.repeat(pr["q"][s][r, b][None], s + 1, axis=0)]))
                seq_k.append(np.concatenate([px["k"][a:e], hk[r, b]], axis=0))
                seq_v.append(np.concatenate([px["v"][a:e], hv[r, b]], axis=0))
                lens.append(e - a + s + 1)
        cu2 = wl.cu_from_lengths(lens)
        o2 = _prefill(to_dev(np.concatenate(seq_q)), to_dev(np.concatenate(seq_k)), to_dev(np.concatenate(seq_v)),
                      i32_dev(cu2), max(lens))
        torch.cuda.synchronize()
        last = from_dev(o2)[cu2[1:] - 1].reshape(R, W, Hq, d)
        assert_parity(got, last, f"step {s + 1}: decode vs last prefill row over prompt ++ history")
        assert_parity(last, want, f"step {s + 1}: last prefill row vs oracle")
    # the prompt K/V was only read
    assert np.array_equal(bits_from_dev(k_pre), k_snapshot)
