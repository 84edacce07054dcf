"""Tolerance rules for comparing the CUDA results with the double oracle.

Test infrastructure, like the rest of oracle/: used by tests/, by
__graft_entry__.smoke() and by bench.py's CPU-baseline leg.

Bars (fused per-token ops, fine-tuning precision targets):
  * fp32 storage:   |gpu - ref| <= 1e-5 * s + 2^-126
  * bf16 outputs:   |gpu - ref| <= 2 * ulp_bf16(ref) + 2^-17 * s
  * fp32 dw (bf16 inputs): |gpu - ref| <= 2e-3 * |ref| + 2^-16 * s
where s is the oracle's condition scale of the element: the sum of the
absolute values of the terms that form it.  For outputs that cannot cancel
(y, h, du) s = |ref| and the bars are exactly "relative 1e-5", "2 bf16 ulps"
and "relative 2e-3".  For outputs that can cancel to ~0 (dx, dg, RoPE, dw)
the s-term is the floor a correct fp32 computation needs.
"""
import numpy as np
import torch


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def bound(ref, scale, dtype: str, kind: str = "out"):
    ref = np.asarray(ref)
    scale = np.abs(ref) if scale is None else np.asarray(scale)
    if dtype == "f32":
        # fp32 carries no relative precision below its smallest normal
        # number 2^-126, so differences under it are not counted
        return 1e-5 * scale + 2.0 ** -126
    if kind == "dw":
        return 2e-3 * np.abs(ref) + 2.0 ** -16 * scale
    return 2.0 * ulp_bf16(ref) + 2.0 ** -17 * scale


def assert_close(name, got, ref, scale=None, dtype="bf16", kind="out"):
    got, ref = f64(got), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    b = bound(ref, scale, dtype, kind)
    err = np.abs(got - ref)
    bad = ~(err <= b)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        rows = [f"{tuple(i)}: gpu={got[tuple(i)]!r} ref={ref[tuple(i)]!r} "
                f"err={err[tuple(i)]:.3e} bound={b[tuple(i)]:.3e}" for i in idx]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements out of "
                             f"tolerance ({dtype}/{kind}):\n  " + "\n  ".join(rows))
    return float((err / np.maximum(b, 1e-300)).max()) if err.size else 0.0


def literal_figures(got, ref, dtype="bf16", kind="out"):
    """The error of `got` against the literal bars, without the condition
    scale: the largest relative error over nonzero references, for bf16
    outputs the largest distance in bf16 ulps of the reference (and a
    histogram of the distances), and how many
    elements exceed the literal bar (relative 1e-5 in fp32, 2 ulps in bf16,
    relative 2e-3 for dw), i.e. needed the condition-scale floor to pass."""
    got, ref = f64(got), np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    nz = ref != 0
    out = {"elements": int(ref.size),
           "max_rel": float((err[nz] / np.abs(ref[nz])).max()) if nz.any() else 0.0}
    if dtype == "f32":
        lit = 1e-5 * np.abs(ref)
    elif kind == "dw":
        lit = 2e-3 * np.abs(ref)
    else:
        u = ulp_bf16(ref)
        d = err / u
        out["max_ulp"] = float(d.max()) if err.size else 0.0
        # how many elements lie how many bf16 ulps of the reference away
        out["ulp_hist"] = {"0": int((d == 0).sum()), "<=0.5": int(((d > 0) & (d <= 0.5)).sum()),
                           "<=1": int(((d > 0.5) & (d <= 1)).sum()),
                           "<=2": int(((d > 1) & (d <= 2)).sum()), ">2": int((d > 2).sum())}
        lit = 2.0 * u
    out["needed_floor"] = int((err > lit).sum())
    return out

