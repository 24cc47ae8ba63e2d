"""The kernel's FMA-pipe exp2 (Cody-Waite reduction + degree-4 minimax
polynomial): the coefficients compiled into the kernel are the ones the
committed Remez fit produces, and their fp32 evaluation -- emulated step by
step as the kernel performs it -- stays within its stated error bound over
the arguments the kernel can produce (x in [-126, 8]; larger negative x is
clamped)."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_forward_12_gb300", "csrc")


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _kernel_coefficients():
    src = open(os.path.join(CSRC, "sm103_primitives.cuh")).read()
    body = src[src.index("float2 exp2_poly2("):]
    body = body[:body.index("\n}\n")]
    vals = [float(v) for v in re.findall(r"make_float2\(([0-9.]+)f, \1f\)", body)]
    # Horner order in the source: c4, c3, c2, c1, c0
    c4, c3, c2, c1, c0 = vals[:5]
    return [c0, c1, c2, c3, c4]


def test_coefficients_are_the_remez_fit():
    mod = _fit_module()
    c, err = mod.remez_relative(4)
    got = _kernel_coefficients()
    assert got[0] == 1.0
    np.testing.assert_allclose(got, np.float32(c).astype(np.float64), rtol=2e-7, atol=0)
    assert err < 4e-6


def test_fp32_evaluation_error_bound():
    mod = _fit_module()
    c = _kernel_coefficients()
    xs = np.concatenate([np.linspace(-126, 8, 1_000_001, dtype=np.float32),
                         np.float32(np.arange(-126, 9)),             # integers: f = 0
                         np.float32(np.arange(-126, 8)) + np.float32(0.5)])  # ties of the rounding
    y = mod.eval_fp32(c, xs).astype(np.float64)
    rel = np.abs(y / np.exp2(xs.astype(np.float64)) - 1)
    assert rel.max() <= 4e-6
    assert np.all(mod.eval_fp32(c, np.float32(np.arange(-10, 9))) == np.exp2(np.arange(-10, 9)))


def test_clamp_below_range():
    mod = _fit_module()
    c = _kernel_coefficients()
    y = mod.eval_fp32(c, np.array([-127.0, -500.0, -np.inf], dtype=np.float32)).astype(np.float64)
    assert np.all(y > 0) and np.all(y <= 2.0 ** -125)
