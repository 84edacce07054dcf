"""The literal-bar report of oracle/tolerance.py on hand-made errors."""
import numpy as np

from oracle.tolerance import literal_figures, ulp_bf16


def test_literal_figures_bf16():
    ref = np.array([1.0, 3.0, -0.5, 0.0])
    u = ulp_bf16(ref)
    got = ref + np.array([1.0, 3.0, 1.0, 0.0]) * u  # 1, 3 and 1 ulps
    got[3] = 1e-6                                   # ref 0: no relative figure
    out = literal_figures(got, ref, dtype="bf16")
    assert out["elements"] == 4
    assert abs(out["max_ulp"] - 1e-6 / u[3]) < 1e-6 * out["max_ulp"]
    assert abs(out["max_rel"] - 3 * u[1] / 3.0) < 1e-15
    # over 2 ulps: the 3-ulp element and the one at a zero reference
    assert out["needed_floor"] == 2


def test_literal_figures_f32_and_dw():
    ref = np.array([2.0, -4.0, 1e-3])
    got = ref * (1 + np.array([5e-6, 2e-5, 0.0]))
    out = literal_figures(got, ref, dtype="f32")
    assert out["needed_floor"] == 1 and "max_ulp" not in out
    assert abs(out["max_rel"] - 2e-5) < 1e-12
    dw = literal_figures(ref * (1 + np.array([1e-3, 3e-3, 0.0])), ref, dtype="bf16", kind="dw")
    assert dw["needed_floor"] == 1 and "max_ulp" not in dw


def test_ulp_histogram():
    ref = np.array([1.0, 1.0, 1.0, 1.0, 1.0])
    u = ulp_bf16(ref)[0]
    got = ref + np.array([0.0, 0.25, 0.75, 1.5, 3.0]) * u
    h = literal_figures(got, ref, dtype="bf16")["ulp_hist"]
    assert h == {"0": 1, "<=0.5": 1, "<=1": 1, "<=2": 1, ">2": 1}
