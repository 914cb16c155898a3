"""Plausible mistakes planted in copies of the FP8 part of the oracle: the pin suite
(tests/test_oracle_fp8_pins.py) must fail on every one of them."""
import types

import pytest

import tests.test_oracle_fp8_pins as pins
from oracle import fp8

MUTATIONS = {
    "exponent bias 8": ("np.ldexp(1.0 + m / 8.0, (e - 7)", "np.ldexp(1.0 + m / 8.0, (e - 8)"),
    "ties away from zero": ("q = np.rint(a / step)", "q = np.floor(a / step + 0.5)"),
    "no saturation": ("a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))", "a = np.where(nan, 0.0, a)"),
    "subnormal step": ("_SUBNORMAL_STEP = 2.0 ** -9", "_SUBNORMAL_STEP = 2.0 ** -10"),
    "sign bit": ("sign = np.where(c & 0x80, -1.0, 1.0)", "sign = np.where(c & 0x40, -1.0, 1.0)"),
    "exponent mask": ("e = (c >> 3) & 0xF", "e = (c >> 3) & 0x7"),
    "code assembly": ("8.0 * (e + 7) + (q - 8.0)", "8.0 * (e + 7) + q"),
    "scale one power too large": ("    s = math.ldexp(1.0, k)\n", "    s = math.ldexp(1.0, k + 1)\n    return s\n"),
}


def _mutant(old, new):
    src = open(fp8.__file__).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("fp8_mutant")
    mod.__dict__["__package__"] = "oracle"
    mod.__dict__["__file__"] = fp8.__file__
    exec(compile(src.replace(old, new), "fp8_mutant", "exec"), mod.__dict__)
    return mod


def _failures(monkeypatch, mod):
    monkeypatch.setattr(pins, "fp8", mod)
    failed = []
    for name in sorted(n for n in dir(pins) if n.startswith("test_")):
        try:
            getattr(pins, name)()
        except pytest.skip.Exception:
            continue
        except Exception:
            failed.append(name)
    return failed


def test_unmutated_copy_passes(monkeypatch):
    assert _failures(monkeypatch, _mutant("E4M3_MAX = 448.0", "E4M3_MAX = 448.0")) == []


@pytest.mark.filterwarnings("ignore::RuntimeWarning")   # a mutant may cast inf to an integer
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_the_mistake(monkeypatch, name):
    old, new = MUTATIONS[name]
    assert _failures(monkeypatch, _mutant(old, new)), f"no pin caught: {name}"
