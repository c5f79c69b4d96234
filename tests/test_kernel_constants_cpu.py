"""The residual weight's polynomial in the CUDA kernels, checked on the CPU.

After a rejection the kernels weight an element by P_t * (1 - 2^delta),
delta = log2(P_d / P_t) <= 0, forming 1 - 2^delta as delta * p(delta) on
[-1/2, 0] (relative precision where the two rows nearly agree).  The
coefficients are read from the kernel source and evaluated the way the
kernels do (fp32, Horner with fused multiply-adds); the reference is
-expm1(delta * ln 2) in fp64.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "speculative_decoding_verification_09_gb300",
                   "csrc", "specverify.cu")


def kernel_coefficients():
    text = open(SRC).read()
    found = dict(re.findall(r"OMC(\d)\s*=\s*(-?[0-9.e+-]+)f", text))
    assert sorted(found) == ["1", "2", "3", "4", "5"], found
    return [np.float32(found[str(j)]) for j in range(1, 6)]


def fp32_one_minus_exp2(c, d):
    d = d.astype(np.float32)
    p = np.full_like(d, c[-1])
    for cj in c[-2::-1]:
        p = (p.astype(np.float64) * d.astype(np.float64) + np.float64(cj)).astype(np.float32)
    return (p.astype(np.float64) * d.astype(np.float64)).astype(np.float32)


def test_polynomial_relative_error_on_its_interval():
    c = kernel_coefficients()
    d = np.linspace(-0.5, 0.0, 200001)[:-1]
    d = np.concatenate([d, -np.logspace(-30, -1, 4001)])  # the range near 0 as well
    got = fp32_one_minus_exp2(c, d).astype(np.float64)
    exact = -np.expm1(d.astype(np.float32).astype(np.float64) * np.log(2.0))
    rel = np.abs(got / exact - 1)
    assert rel.max() < 2e-7, rel.max()


def test_polynomial_is_zero_at_zero_and_positive_below():
    c = kernel_coefficients()
    assert fp32_one_minus_exp2(c, np.array([0.0]))[0] == 0.0
    d = -np.logspace(-38, np.log10(0.5), 1000)
    assert (fp32_one_minus_exp2(c, d) > 0).all()


def test_polynomial_meets_the_alternative_at_the_switch():
    # at delta = -1/2 the kernels switch to 1 - ex2(delta); both sides agree there
    c = kernel_coefficients()
    v = fp32_one_minus_exp2(c, np.array([-0.5]))[0]
    assert abs(v / (1 - 2 ** -0.5) - 1) < 2e-7
