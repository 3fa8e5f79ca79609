"""The exp2 polynomial of the attention kernels' softmax (part of the
exponentials run on the FMA pipe): its constants are the Remez fit of
exp2_poly.py, and its error, evaluated with the kernels' fp32 steps, stays
far below the bf16 resolution of P (2^-9) and keeps the row sum, hence the
LSE, within 1e-4 relative."""
import os
import re

import numpy as np

from varlen_flashattention_forward_gb300 import exp2_poly

KERNEL = os.path.join(os.path.dirname(exp2_poly.__file__), "csrc", "varlen_fwd_kernel.cuh")


def kernel_constants():
    text = open(KERNEL).read()
    vals = {int(m.group(1)): float(m.group(2))
            for m in re.finditer(r"constexpr float kExp2C(\d) = ([-+0-9.e]+)f;", text)}
    return np.array([vals[k] for k in range(4)], dtype=np.float32)


def test_kernel_constants_are_the_remez_fit():
    c, E = exp2_poly.remez()
    fit = exp2_poly.fp32_coefficients(c)
    got = kernel_constants()
    # The kernel holds the fp32 roundings printed with 10 significant digits.
    assert np.all(np.abs(got - fit) <= np.abs(fit) * 2.0 ** -23), (got, fit)
    assert 7e-5 < E < 8e-5


def test_error_bound_in_fp32():
    c32 = kernel_constants()
    err = exp2_poly.max_rel_error(c32)
    assert err < 7.6e-5
    assert err < 2.0 ** -9 / 20  # twenty times below a bf16 rounding step


def test_equioscillation_of_the_fit():
    # A minimax fit's error reaches its maximum with alternating signs at
    # degree + 2 points; a wrong coefficient breaks the alternation.
    c, E = exp2_poly.remez()
    f = np.linspace(-0.5, 0.5, 100001)
    err = np.polyval(c[::-1], f) / 2.0 ** f - 1.0
    near = np.abs(np.abs(err) - E) < 1e-3 * E
    signs = np.sign(err[near])
    changes = int(np.sum(signs[1:] != signs[:-1]))
    assert changes >= exp2_poly.DEGREE + 1


def test_range_ends_and_integers():
    c32 = kernel_constants()
    x = np.array([-125.0, -100.5, -1.0, -0.5, 0.0, 0.49, 3.0, 8.0], dtype=np.float32)
    got = exp2_poly.eval_fp32(c32, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.all(np.isfinite(got)) and np.all(got > 0)
    assert np.all(np.abs(got / ref - 1) < 7.6e-5)
    # Below the clamp the value stays the (normal) 2^-125 scale, never
    # wrapping the exponent.
    tiny = exp2_poly.eval_fp32(c32, np.array([-1e4, -126.0], dtype=np.float32))
    assert np.all(tiny > 0) and np.all(tiny < 2.0 ** -124)
