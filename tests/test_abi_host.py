"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/bg_attn.h declares, and rejects bad arguments before
enqueuing anything."""
import ctypes
import os
import re

import pytest

from attention_packed_varlen_causal_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bg_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("bg_packed_prefill_attn", "bg_beam_decode_attn", "bg_beam_suffix_reorder",
              "bg_packed_prefill_workspace_size", "bg_status_string"):
        assert n in names


def header_constants():
    """Every #define with a numeric value and every bg_status_t enumerator in bg_attn.h."""
    text = open(os.path.join(ROOT, "include", "bg_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    vals = {}
    for name, expr in re.findall(r"#define[ \t]+(BG_[A-Z0-9_]+)[ \t]+([^\n]+)", text):
        expr = re.sub(r"(?<=\d)u\b", "", expr.strip())       # 1u -> 1
        vals[name] = int(eval(expr, {"__builtins__": {}}))    # literals and shifts only
    for name, v in re.findall(r"\b(BG_[A-Z_]+)\s*=\s*(\d+)", text):
        vals[name] = int(v)
    return vals


def test_binding_constants_match_the_header():
    vals = header_constants()
    assert len(vals) >= 15
    for name, v in vals.items():
        assert hasattr(binding, name), f"{name} is defined in bg_attn.h but not in the binding"
        assert getattr(binding, name) == v, f"{name}: header {v}, binding {getattr(binding, name)}"


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in bg_attn.h but not exported"
        assert n in binding.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(lib):
    assert binding.status_string(0) == "BG_OK"
    assert binding.status_string(1) == "BG_ERR_INVALID_ARG"
    assert binding.status_string(99) == "BG_ERR_UNKNOWN"


def test_workspace_size(lib):
    ws = lib.bg_packed_prefill_workspace_size(240, 70375, 500, 16, 8, 128)
    assert ws % 256 == 0 and ws >= 256 + 16 * (70375 // 128 + 240)
    assert lib.bg_packed_prefill_workspace_size(-1, 5, 5, 1, 1, 64) == 0


FAKE = 0x10000          # 16-byte aligned, never dereferenced: every call below fails validation first


def prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, cu=FAKE * 4, B=2, T=10, maxlen=8, Hq=4, Hkv=2, d=64, scale=0.125,
             out=FAKE * 5, lse=None, ws=FAKE * 6, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    return lib.bg_packed_prefill_attn(a["q"], a["k"], a["v"], a["cu"], a["B"], a["T"], a["maxlen"], a["Hq"],
                                      a["Hkv"], a["d"], a["scale"], a["out"], a["lse"], a["ws"], a["wsb"], a["st"],
                                      a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(cu=None), 1), (dict(out=None), 1), (dict(ws=None), 1),
    (dict(Hq=6, Hkv=4), 1), (dict(d=96), 2), (dict(d=256), 2), (dict(maxlen=70000), 2),
    (dict(B=-1), 1), (dict(q=FAKE + 8), 1), (dict(ws=FAKE * 6 + 16), 1), (dict(wsb=64), 1),
    (dict(out=FAKE * 1 + 64), 1),            # out overlaps q
    (dict(scale=float("nan")), 1), (dict(scale=0.0), 1), (dict(scale=-0.125), 1),
    (dict(B=0, q=None), 0), (dict(T=0, q=None), 0),   # empty problems are a no-op
])
def test_prefill_host_validation(lib, kw, expect):
    assert prefill(lib, **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(cu=None), 1), (dict(out=None), 1), (dict(ws=None), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(d=96), 2), (dict(maxlen=70000), 2), (dict(wsb=64), 1), (dict(out=FAKE * 1 + 64), 1),
    (dict(scale=0.0), 1), (dict(B=0, q=None), 0),
])
def test_prefill_planned_host_validation(lib, kw, expect):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, cu=FAKE * 4, B=2, T=10, maxlen=8, Hq=4, Hkv=2, d=64, scale=0.125,
             out=FAKE * 5, lse=None, ws=FAKE * 6, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    assert lib.bg_packed_prefill_attn_planned(a["q"], a["k"], a["v"], a["cu"], a["B"], a["T"], a["maxlen"], a["Hq"],
                                              a["Hkv"], a["d"], a["scale"], a["out"], a["lse"], a["ws"], a["wsb"],
                                              a["st"], a["stream"]) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(cu=None), 1), (dict(ws=None), 1), (dict(wsb=64), 1), (dict(maxlen=70000), 2), (dict(B=-1), 1),
    (dict(T=-1), 1), (dict(cu=FAKE * 4 + 2), 1), (dict(ws=FAKE * 6 + 16), 1), (dict(st=FAKE * 7 + 2), 1),
    (dict(cu=FAKE * 6 + 256), 1),               # cu_seqlens inside the workspace
    (dict(B=0, cu=None), 0), (dict(T=0, cu=None), 0),   # empty packings are a no-op
])
def test_prefill_plan_host_validation(lib, kw, expect):
    a = dict(cu=FAKE * 4, B=2, T=10, maxlen=8, ws=FAKE * 6, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    assert lib.bg_packed_prefill_plan(a["cu"], a["B"], a["T"], a["maxlen"], a["ws"], a["wsb"], a["st"],
                                      a["stream"]) == expect


def prefill_fp8(lib, **kw):
    a = dict(q=FAKE, qs=0.5, k=FAKE * 2, ks=0.25, v=FAKE * 3, cu=FAKE * 4, B=2, T=10, maxlen=8, Hq=4, Hkv=2, d=128,
             scale=0.125, out=FAKE * 5, lse=None, ws=FAKE * 6, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    return lib.bg_packed_prefill_attn_fp8(a["q"], a["qs"], a["k"], a["ks"], a["v"], a["cu"], a["B"], a["T"],
                                          a["maxlen"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["out"], a["lse"],
                                          a["ws"], a["wsb"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(ws=None), 1), (dict(wsb=64), 1),
    (dict(qs=0.0), 1), (dict(ks=-1.0), 1), (dict(qs=float("inf")), 1), (dict(ks=float("nan")), 1),
    (dict(qs=1e30, ks=1e30), 1),                    # the folded scale overflows
    (dict(d=64), 2), (dict(d=96), 2), (dict(Hq=6, Hkv=4), 1), (dict(scale=0.0), 1),
    (dict(out=FAKE * 1 + 64), 1),                   # out overlaps the codes of q
    (dict(B=0, q=None), 0),
])
def test_prefill_fp8_host_validation(lib, kw, expect):
    assert prefill_fp8(lib, **kw) == expect


def last_token(lib, **kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, cu=FAKE * 4, B=2, T=10, maxlen=8, Hq=4, Hkv=2, d=64, scale=0.125,
             out=FAKE * 5, lse=None, st=None, stream=None)
    a.update(kw)
    return lib.bg_packed_last_token_attn(a["q"], a["k"], a["v"], a["cu"], a["B"], a["T"], a["maxlen"], a["Hq"],
                                         a["Hkv"], a["d"], a["scale"], a["out"], a["lse"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(cu=None), 1), (dict(out=None), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(d=96), 2), (dict(maxlen=70000), 2), (dict(Hq=34, Hkv=2), 2), (dict(q=FAKE + 8), 1),
    (dict(out=FAKE * 2), 1), (dict(lse=FAKE * 5 + 4), 1), (dict(scale=0.0), 1), (dict(B=-1), 1),
    (dict(B=0, q=None), 0),
])
def test_last_token_host_validation(lib, kw, expect):
    assert last_token(lib, **kw) == expect


def decode(lib, **kw):
    a = dict(q=FAKE, pk=FAKE * 2, pv=FAKE * 3, cu=FAKE * 4, P=100, maxP=60, sk=FAKE * 8, sv=FAKE * 16, t=2, S=4,
             R=2, W=5, Hq=14, Hkv=2, d=64, scale=0.125, out=FAKE * 32, st=None, stream=None)
    a.update(kw)
    return lib.bg_beam_decode_attn(a["q"], a["pk"], a["pv"], a["cu"], a["P"], a["maxP"], a["sk"], a["sv"], a["t"],
                                   a["S"], a["R"], a["W"], a["Hq"], a["Hkv"], a["d"], a["scale"], a["out"], a["st"],
                                   a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(cu=None), 1), (dict(t=5), 1), (dict(t=-1), 1),
    (dict(pk=None), 1), (dict(sk=None), 1), (dict(Hq=15), 1), (dict(d=80), 2), (dict(S=17, t=2), 2),
    (dict(Hq=258, Hkv=2), 2), (dict(maxP=0, t=0), 1), (dict(W=0), 1), (dict(out=FAKE + 16), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1),
    (dict(R=0, q=None), 0),
])
def test_decode_host_validation(lib, kw, expect):
    assert decode(lib, **kw) == expect


def reorder(lib, **kw):
    a = dict(sk=FAKE, sv=FAKE * 2, dk=FAKE * 4, dv=FAKE * 8, par=FAKE * 16, nk=None, nv=None, R=2, W=3, S=4, n=2,
             Hkv=2, d=64, st=None, stream=None)
    a.update(kw)
    return lib.bg_beam_suffix_reorder(a["sk"], a["sv"], a["dk"], a["dv"], a["par"], a["nk"], a["nv"], a["R"],
                                      a["W"], a["S"], a["n"], a["Hkv"], a["d"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(sk=None), 1), (dict(par=None), 1), (dict(n=5), 1), (dict(n=4, nk=FAKE * 32, nv=FAKE * 64), 1),
    (dict(nk=FAKE * 32), 1), (dict(dk=FAKE), 1), (dict(dk=FAKE * 2 + 256), 1), (dict(d=32), 2),
    (dict(sk=FAKE + 4), 1), (dict(W=0), 1), (dict(R=0, sk=None), 0),
])
def test_reorder_host_validation(lib, kw, expect):
    assert reorder(lib, **kw) == expect


def step(lib, **kw):
    a = dict(q=FAKE, pk=FAKE * 2, pv=FAKE * 3, cu=FAKE * 4, P=100, maxP=60, sk=FAKE * 8, sv=FAKE * 16,
             par=FAKE * 24, nk=FAKE * 32, nv=FAKE * 40, dk=FAKE * 48, dv=FAKE * 56, t=2, S=4, R=2, W=5, Hq=14, Hkv=2,
             d=64, scale=0.125, out=FAKE * 64, st=None, stream=None)
    a.update(kw)
    return lib.bg_beam_decode_step(a["q"], a["pk"], a["pv"], a["cu"], a["P"], a["maxP"], a["sk"], a["sv"], a["par"],
                                   a["nk"], a["nv"], a["dk"], a["dv"], a["t"], a["S"], a["R"], a["W"], a["Hq"],
                                   a["Hkv"], a["d"], a["scale"], a["out"], a["st"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(t=0), 1), (dict(t=5), 1), (dict(par=None), 1), (dict(nk=None), 1), (dict(nv=None), 1),
    (dict(sk=None), 1),                                  # t = 2 moves one slot: src is needed
    (dict(dk=FAKE * 8), 1),                              # dst is src
    (dict(dk=FAKE), 1), (dict(dv=FAKE * 2 + 256), 1),    # dst inside q / the prompt K
    (dict(dv=FAKE * 48 + 256), 1),                       # dst K and V overlap
    (dict(dk=FAKE * 24), 1), (dict(dk=FAKE * 32), 1),    # dst over the parents / the new token
    (dict(out=FAKE * 24), 1), (dict(out=FAKE * 40), 1),  # out over the parents / the new token
    (dict(par=FAKE * 24 + 2), 1), (dict(nk=FAKE * 32 + 8), 1), (dict(sk=FAKE * 8 + 8), 1),
    (dict(d=32), 2), (dict(S=17, t=2), 2), (dict(Hq=15), 1), (dict(R=0), 0),
])
def test_decode_step_host_validation(lib, kw, expect):
    assert step(lib, **kw) == expect


def test_selftest_host_checks(lib):
    assert lib.bg_selftest_wait_timeout(None, FAKE, None) == binding.BG_ERR_INVALID_ARG
    assert lib.bg_selftest_wait_timeout(FAKE, None, None) == binding.BG_ERR_INVALID_ARG
    assert lib.bg_selftest_wait_timeout(FAKE + 2, FAKE * 2, None) == binding.BG_ERR_INVALID_ARG
    assert lib.bg_selftest_wait_timeout(FAKE, FAKE * 2 + 4, None) == binding.BG_ERR_INVALID_ARG


def test_beam_select_host_checks(lib):
    ws = lib.bg_beam_select_workspace_size(32, 100, 65536)
    assert ws % 256 == 0 and ws >= 32 * 100 * 100 * 8 + 32 * 100 * 4
    assert lib.bg_beam_select_workspace_size(-1, 4, 8) == 0

    def sel(**kw):
        a = dict(logits=FAKE, cum=FAKE * 2, R=2, W=4, V=16, tok=FAKE * 3, par=FAKE * 4, sc=FAKE * 5, ws=FAKE * 6,
                 wsb=1 << 20)
        a.update(kw)
        return lib.bg_beam_select(a["logits"], a["cum"], a["R"], a["W"], a["V"], a["tok"], a["par"], a["sc"],
                                  a["ws"], a["wsb"], None)

    assert sel(R=0) == binding.BG_OK                         # nothing to do, nothing launched
    assert sel(R=-1) == binding.BG_ERR_INVALID_ARG
    assert sel(W=0) == binding.BG_ERR_UNSUPPORTED
    assert sel(W=binding.BG_MAX_BEAM + 1, V=1 << 20) == binding.BG_ERR_UNSUPPORTED
    assert sel(V=3) == binding.BG_ERR_UNSUPPORTED            # fewer tokens than beams
    assert sel(V=binding.BG_MAX_VOCAB + 1) == binding.BG_ERR_UNSUPPORTED
    assert sel(logits=None) == binding.BG_ERR_INVALID_ARG
    assert sel(tok=None) == binding.BG_ERR_INVALID_ARG
    assert sel(logits=FAKE + 4) == binding.BG_ERR_INVALID_ARG   # logits need 16-byte alignment
    assert sel(ws=FAKE + 16) == binding.BG_ERR_INVALID_ARG     # workspace needs 256-byte alignment
    assert sel(wsb=16) == binding.BG_ERR_INVALID_ARG
    assert sel(tok=FAKE * 8 + 64, logits=FAKE * 8) == binding.BG_ERR_INVALID_ARG   # output inside the logits
    assert sel(par=FAKE * 3) == binding.BG_ERR_INVALID_ARG               # two outputs overlap


_NOALLOC_CHECK = r"""
import sys
from attention_packed_varlen_causal_gb300 import binding as bg
lib = bg.load()
fake = 1 << 32          # 4 GiB apart: the tensors these sizes describe do not overlap
def call(num_seqs, total, Hq, Hkv, q=fake):
    return lib.bg_packed_prefill_attn_noalloc(q, fake * 2, fake * 3, fake * 4, num_seqs, total, 1, Hq, Hkv, 128,
                                              0.1, fake * 5, None, None, None)
# 200,000 sequences need more work-list entries than the fixed scratch holds
print(call(200000, 200000, 16, 8),   # valid but too large
      call(200000, 200000, 16, 7),   # Hq % Hkv != 0: the argument error wins over the size
      call(200000, 200000, 16, 8, q=None))
"""


def test_noalloc_host_checks_run_in_order_without_a_device():
    """bg_packed_prefill_attn_noalloc checks its arguments first (bad ones give
    BG_ERR_INVALID_ARG whatever the size), then rejects a valid problem whose work list
    does not fit its fixed scratch with BG_ERR_UNSUPPORTED, both before any CUDA call.
    The calls run in a child process that sees no GPU, so even a regression of these
    checks cannot launch anything on fake pointers: it would come back as BG_ERR_CUDA."""
    import subprocess
    import sys
    build.build()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _NOALLOC_CHECK], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    codes = [int(c) for c in r.stdout.split()]
    assert codes == [binding.BG_ERR_UNSUPPORTED, binding.BG_ERR_INVALID_ARG, binding.BG_ERR_INVALID_ARG]
