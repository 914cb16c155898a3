"""Runs one hot-path call on a named workload a few times, for profilers.

    python profile_case.py prefill_only --iters 3
    python profile_case.py beam_long --iters 2
    python profile_case.py beam_long --iters 2 --two-call
    python profile_case.py select_long --iters 2
    python profile_case.py prefill_only --iters 3 --fp8

Prefill workloads (tiny, prefill_only, skewed) call bg_packed_prefill_attn
``iters`` times on one layer of inputs; decode workloads (beam_short,
beam_long) run ``iters`` complete beam searches of one layer (per step the
suffix reorder + append, then the decode attention: one bg_beam_decode_step
call, or with ``--two-call`` bg_beam_suffix_reorder, then
bg_beam_decode_attn); selection workloads
(select_short, select_long) call bg_beam_select ``iters`` times on the beam
configurations' shapes with fp32 logits N(0, 3) over 65,536 tokens.  Inputs are drawn on the
device with a seeded generator, shaped as in ``workloads``.  Nothing is
timed here: use ncu (or bench.py for timings).
"""
from __future__ import annotations

import argparse
import math
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import numpy as np
    import torch

    from attention_packed_varlen_causal_gb300 import binding as bg
    from attention_packed_varlen_causal_gb300 import build
    from attention_packed_varlen_causal_gb300 import workloads as wl

    ap = argparse.ArgumentParser()
    select = {"select_short": "beam_short", "select_long": "beam_long"}
    ap.add_argument("workload", choices=sorted(list(wl.PREFILL_CONFIGS) + list(wl.DECODE_CONFIGS) + list(select)))
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--two-call", action="store_true", help="decode: separate reorder and attention calls")
    ap.add_argument("--fp8", action="store_true", help="prefill: E4M3 Q and K (bg_packed_prefill_attn_fp8)")
    args = ap.parse_args(argv)
    build.build()
    bg.load()
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    bf = torch.bfloat16
    if args.workload in select:
        cfg = wl.DECODE_CONFIGS[select[args.workload]]
        R, W, V = cfg.R, cfg.W, 65536
        logits = torch.randn((R, W, V), generator=g, device=dev) * 3.0
        cum = torch.randn((R, W), generator=g, device=dev) - 3.0
        tok = torch.empty((R, W), dtype=torch.int32, device=dev)
        par = torch.empty_like(tok)
        sc = torch.empty((R, W), dtype=torch.float32, device=dev)
        ws = torch.empty(bg.bg_beam_select_workspace_size(R, W, V), dtype=torch.uint8, device=dev)
        for _ in range(args.iters):
            bg.bg_beam_select(logits, cum, tok, par, sc, workspace=ws)
    elif args.workload in wl.PREFILL_CONFIGS:
        cfg = wl.PREFILL_CONFIGS[args.workload]
        lengths = wl.prefill_lengths(cfg)
        cu_np = wl.cu_from_lengths(lengths)
        T = int(cu_np[-1])
        q = torch.randn((T, cfg.Hq, cfg.head_dim), generator=g, device=dev).to(bf)
        k = torch.randn((T, cfg.Hkv, cfg.head_dim), generator=g, device=dev).to(bf)
        v = torch.randn((T, cfg.Hkv, cfg.head_dim), generator=g, device=dev).to(bf)
        out = torch.empty_like(q)
        cu = torch.from_numpy(cu_np).to(dev)
        ws = torch.empty(bg.bg_packed_prefill_workspace_size(len(lengths), T, max(lengths), cfg.Hq, cfg.Hkv,
                                                             cfg.head_dim), dtype=torch.uint8, device=dev)
        if args.fp8:
            # E4M3 codes of q and k with one power-of-two scale each (max |x| / scale <= 448)
            codes = []
            for x in (q, k):
                s8 = 2.0 ** math.ceil(math.log2(float(x.abs().max().float().item()) / 448.0))
                codes.append(((x.float() / s8).to(torch.float8_e4m3fn).view(torch.uint8), s8))
            for _ in range(args.iters):
                bg.bg_packed_prefill_attn_fp8(codes[0][0], codes[0][1], codes[1][0], codes[1][1], v, cu, max(lengths),
                                              out, workspace=ws)
        else:
            for _ in range(args.iters):
                bg.bg_packed_prefill_attn(q, k, v, cu, max(lengths), out, workspace=ws)
    else:
        cfg = wl.DECODE_CONFIGS[args.workload]
        plen = wl.decode_prompt_lengths(cfg)
        cu_np = wl.cu_from_lengths(plen)
        P = int(cu_np[-1])
        R, W, Hq, Hkv, d, S = cfg.R, cfg.W, cfg.Hq, cfg.Hkv, cfg.head_dim, cfg.steps
        pk = torch.randn((P, Hkv, d), generator=g, device=dev).to(bf)
        pv = torch.randn((P, Hkv, d), generator=g, device=dev).to(bf)
        cu = torch.from_numpy(cu_np).to(dev)
        qs = [torch.randn((R, W, Hq, d), generator=g, device=dev).to(bf) for _ in range(S)]
        nk = [torch.randn((R, W, Hkv, d), generator=g, device=dev).to(bf) for _ in range(S)]
        nv = [torch.randn((R, W, Hkv, d), generator=g, device=dev).to(bf) for _ in range(S)]
        parents = [torch.from_numpy(np.random.default_rng(wl.SEED_PARENT + s).integers(0, W, size=(R, W))
                                    .astype(np.int32)).to(dev) for s in range(S)]
        sk = [torch.zeros((R, W, S, Hkv, d), dtype=bf, device=dev) for _ in range(2)]
        sv = [torch.zeros((R, W, S, Hkv, d), dtype=bf, device=dev) for _ in range(2)]
        out = torch.empty_like(qs[0])
        for _ in range(args.iters):
            for s in range(S):
                src, dst = s % 2, 1 - s % 2
                if not args.two_call:
                    bg.bg_beam_decode_step(qs[s], pk, pv, cu, max(plen), sk[src], sv[src], parents[s], nk[s], nv[s],
                                           sk[dst], sv[dst], s + 1, out)
                    continue
                bg.bg_beam_suffix_reorder(sk[src], sv[src], sk[dst], sv[dst], parents[s], s, new_k=nk[s],
                                          new_v=nv[s])
                bg.bg_beam_decode_attn(qs[s], pk, pv, cu, max(plen), sk[dst], sv[dst], s + 1, out)
    torch.cuda.synchronize()
    print(f"profile_case {args.workload}: {args.iters} iteration(s) done")


if __name__ == "__main__":
    main()
