"""Plants plausible mistakes in copies of oracle/beam_select.py (on the CPU) and
checks that the pins in test_oracle_select_pins.py catch every one."""
import importlib.util
import os

import pytest

from tests.test_oracle_select_pins import CHECKS

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "beam_select.py")

# (name, exact text in beam_select.py, replacement)
MUTATIONS = [
    ("logsumexp dropped", "return x - (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))", "return x"),
    ("max not added back", "return x - (m + np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True)))",
     "return x - np.log(np.sum(np.exp(x - m), axis=-1, keepdims=True))"),
    ("accumulated score ignored", "s = (c[r][:, None] + lp[r]).reshape(-1)", "s = lp[r].reshape(-1)"),
    ("accumulated score subtracted", "s = (c[r][:, None] + lp[r]).reshape(-1)", "s = (lp[r] - c[r][:, None]).reshape(-1)"),
    ("ties: larger index first", "order = np.lexsort((flat_index, -s))", "order = np.lexsort((-flat_index, -s))"),
    ("lowest scores kept", "order = np.lexsort((flat_index, -s))", "order = np.lexsort((flat_index, s))"),
    ("parent and token swapped", "parent[r] = (keep // V).astype(np.int32)\n        token[r] = (keep % V).astype(np.int32)",
     "parent[r] = (keep % V).astype(np.int32)\n        token[r] = (keep // V).astype(np.int32)"),
    ("best candidate dropped", "keep = order[:W]", "keep = order[1:W + 1]"),
    ("per-beam selection without merge", "keep = order[:W]",
     "keep = np.array([b * V + int(np.argmax(s[b * V:(b + 1) * V])) for b in range(W)])"),
]


def _load_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    path = tmp_path / "beam_select_mut.py"
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("beam_select_mut", str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_select_pins_catch_planted_mistake(tmp_path, name, old, new):
    mod = _load_mutant(tmp_path, old, new)
    caught = []
    for check in CHECKS:
        try:
            check(mod)
        except Exception:   # an assertion or a crash of the mutant: the pin caught it
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
