"""Plants plausible mistakes in copies of the oracle (on the CPU only) and
checks that the pin suite in test_oracle_pins.py catches every one of them."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTATIONS = [
    ("causal sees one future key", "keys, vals, p + 1, d", "keys, vals, (p + 2 > L ? L : p + 2), d"),
    ("causal drops the diagonal", "keys, vals, p + 1, d", "keys, vals, (p > 0 ? p : 1), d"),
    ("gqa head mapping modulo", "const int32_t kh = h / g;\n                const int64_t s0", "const int32_t kh = h % Hkv;\n                const int64_t s0"),
    ("scale dropped", "z[j] = scale * dot;", "z[j] = dot;"),
    ("values read from keys", "acc += z[j] * bf16_to_double(vals[j][c]);", "acc += z[j] * bf16_to_double(keys[j][c]);"),
    ("softmax not normalised", "out[c] = acc / den;", "out[c] = acc / (den + 0.5);"),
    ("sequence offset ignored", "const int64_t s0 = cu[i];", "const int64_t s0 = cu[i] > 0 ? cu[i] - 1 : 0;"),
    ("decode prompt offset ignored", "keys[j] = pk + ((p0 + j) * Hkv + kh) * d;", "keys[j] = pk + ((j) * Hkv + kh) * d;"),
    ("decode suffix order lost", "keys[P + s] = hk + ((rb * t + s) * Hkv + kh) * d;", "keys[P + s] = hk + ((rb * t + 0) * Hkv + kh) * d;"),
    ("last token drops its own key", "keys, vals, L, d, scale, z,", "keys, vals, (L > 1 ? L - 1 : 1), d, scale, z,"),
    ("last token reads the wrong query head", "attend_row(q + ((int64_t)i * Hq + h) * d,",
     "attend_row(q + ((int64_t)i * Hq + (h ^ 1)) * d,"),
    ("decode prompt dropped", "attend_row(q + (rb * Hq + h) * d, keys, vals, P + t,", "attend_row(q + (rb * Hq + h) * d, keys + P, vals + P, t > 0 ? t : P,"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "oracle_mut.c"
    so_path = tmp_path / "liboracle_mut.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c99", str(c_path), "-o", str(so_path), "-lm"],
                   check=True)
    env = dict(os.environ, BG_ORACLE_LIB=str(so_path), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' was not caught by any pin:\n{r.stdout[-2000:]}"


def test_pins_catch_history_without_parent(monkeypatch):
    """Reorder mistake planted in the Python history: beams keep their own
    history instead of their parent's."""
    import numpy as np
    import oracle

    def bad_step(self, parent, new_k=None, new_v=None):
        nxt = []
        for r in range(self.R):
            row = []
            for b in range(self.W):
                h = list(self.rows[r][b])
                if new_k is not None:
                    h.append((np.array(new_k[r, b]), np.array(new_v[r, b])))
                row.append(h)
            nxt.append(row)
        self.rows = nxt

    monkeypatch.setattr(oracle.BeamHistory, "step", bad_step)
    from tests import test_oracle_pins as pins
    with pytest.raises(AssertionError):
        pins.test_history_follows_parent_chain()
