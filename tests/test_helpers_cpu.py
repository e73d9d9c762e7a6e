"""CPU checks of the test helpers that the GPU tests rely on (no device needed)."""
import numpy as np
import pytest

from helpers import compare_chain_runs

SPEC = [("x0", [("a", 8, 4)]), ("a", [("b", 4, 4)])]


def runs(seed=0):
    rng = np.random.default_rng(seed)
    first = {n: rng.standard_normal(4).astype(np.float16) for n in ("x0", "a", "b")}
    return first, {k: v.copy() for k, v in first.items()}


def bump(v, i, n):
    """v with element i moved by n fp16 ulps."""
    out = v.copy()
    out[i] = np.float16(np.float64(v[i]) + n * np.float64(np.spacing(np.abs(v[i]))))
    return out


def test_identical_runs_compare_every_link():
    first, second = runs()
    assert compare_chain_runs(first, second, SPEC) == ["x0", "a"]


def test_last_place_differences_pass_and_large_ones_fail():
    first, second = runs(1)
    second["a"] = bump(first["a"], 0, 2)  # a differs by 2 ulp: within 8
    assert compare_chain_runs(first, second, SPEC) == ["x0"]  # link b's input now differs
    second["a"] = bump(first["a"], 0, 40)
    with pytest.raises(AssertionError):
        compare_chain_runs(first, second, SPEC)


def test_link_with_a_differing_input_is_not_compared():
    first, second = runs(2)
    second["a"] = bump(first["a"], 1, 1)
    second["b"] = first["b"] + np.float16(1.0)  # far apart, but its input differs
    assert compare_chain_runs(first, second, SPEC) == ["x0"]
