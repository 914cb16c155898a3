"""bg_beam_suffix_reorder on the GPU: bit-exact gather by parent index, with
and without the append, against a numpy gather of the same bits."""
import numpy as np
import pytest

from attention_packed_varlen_causal_gb300 import binding as bg
from attention_packed_varlen_causal_gb300 import build
from tests.helpers import bits_from_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    bg.load()


@pytest.mark.parametrize("R,W,S,n,Hkv,d,append", [
    (32, 100, 4, 3, 2, 64, True), (16, 400, 5, 4, 2, 64, False), (3, 7, 6, 0, 4, 128, True),
    (1, 1, 1, 1, 1, 64, False), (5, 33, 16, 15, 1, 128, True),
])
def test_reorder_bitexact(R, W, S, n, Hkv, d, append):
    import torch
    rng = np.random.default_rng(R * 1000 + W)
    src_k = rng.integers(0, 65536, size=(R, W, S, Hkv, d), dtype=np.uint16)
    src_v = rng.integers(0, 65536, size=(R, W, S, Hkv, d), dtype=np.uint16)
    parent = rng.integers(0, W, size=(R, W)).astype(np.int32)
    new_k = rng.integers(0, 65536, size=(R, W, Hkv, d), dtype=np.uint16)
    new_v = rng.integers(0, 65536, size=(R, W, Hkv, d), dtype=np.uint16)
    dk = torch.full((R, W, S, Hkv, d), 0x1234, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dv = torch.full((R, W, S, Hkv, d), 0x1234, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    bg.bg_beam_suffix_reorder(to_dev(src_k), to_dev(src_v), dk, dv, i32_dev(parent), n,
                              new_k=to_dev(new_k) if append else None, new_v=to_dev(new_v) if append else None)
    torch.cuda.synchronize()
    gk, gv = bits_from_dev(dk), bits_from_dev(dv)
    exp_k = np.full_like(src_k, 0x1234)
    exp_v = np.full_like(src_v, 0x1234)
    for r in range(R):
        exp_k[r, :, :n] = src_k[r, parent[r], :n]
        exp_v[r, :, :n] = src_v[r, parent[r], :n]
        if append:
            exp_k[r, :, n] = new_k[r]
            exp_v[r, :, n] = new_v[r]
    np.testing.assert_array_equal(gk, exp_k)
    np.testing.assert_array_equal(gv, exp_v)


def test_identity_parent_and_composition():
    import torch
    R, W, S, Hkv, d = 4, 50, 4, 2, 64
    rng = np.random.default_rng(3)
    k0 = rng.integers(0, 65536, size=(R, W, S, Hkv, d), dtype=np.uint16)
    buf = [to_dev(k0), torch.empty_like(to_dev(k0)), torch.empty_like(to_dev(k0))]
    vbuf = [to_dev(k0), torch.empty_like(buf[0]), torch.empty_like(buf[0])]
    ident = np.tile(np.arange(W, dtype=np.int32), (R, 1))
    bg.bg_beam_suffix_reorder(buf[0], vbuf[0], buf[1], vbuf[1], i32_dev(ident), S)
    p1 = rng.integers(0, W, size=(R, W)).astype(np.int32)
    p2 = rng.integers(0, W, size=(R, W)).astype(np.int32)
    bg.bg_beam_suffix_reorder(buf[1], vbuf[1], buf[2], vbuf[2], i32_dev(p1), S)
    bg.bg_beam_suffix_reorder(buf[2], vbuf[2], buf[1], vbuf[1], i32_dev(p2), S)
    torch.cuda.synchronize()
    comp = np.take_along_axis(p1, p2, axis=1)
    got = bits_from_dev(buf[1])
    for r in range(R):
        np.testing.assert_array_equal(got[r], k0[r][comp[r]])
