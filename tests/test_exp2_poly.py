"""The FMA-pipe exp2 used for part of the softmax exponentials.

Checks that the coefficients compiled into the kernel are the ones the
committed Remez fit produces, and that the kernel's sequence of float32
operations (Cody-Waite reduction to the nearest integer, degree-3 minimax
polynomial, exponent add) stays within 2e-4 relative error of the exact
2^x over [-125, 8] (the reference max may trail the true max by up to 2^8,
so arguments reach 8; below -125 only tiny non-negative values are needed).
"""
from __future__ import annotations

import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dynamic_block_sparse_causal_gb300", "csrc")


def fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def kernel_coeffs():
    src = open(os.path.join(CSRC, "bsa_fwd.cu")).read()
    got = {}
    for name, val in re.findall(r"kExp2C(\d)\s*=\s*([-+0-9.eE]+)f", src):
        got[int(name)] = float(np.float32(val))
    return [got[i] for i in range(4)]


def test_kernel_coefficients_are_the_fit():
    m = fit_module()
    assert kernel_coeffs() == m.f32_coeffs(m.remez())


def test_emulated_exp2_error_bound():
    m = fit_module()
    c = kernel_coeffs()
    xs = np.concatenate([np.linspace(-125.0, 8.0, 1000001, dtype=np.float32),
                         np.float32(np.arange(-125, 9)),          # exact integers
                         np.float32(np.arange(-125, 8)) + np.float32(0.5)])
    got = m.emulate(xs, c).astype(np.float64)
    rel = np.abs(got / np.exp2(xs.astype(np.float64)) - 1.0)
    assert rel.max() < 2e-4
    # far below the range: tiny and non-negative, never NaN / negative
    low = m.emulate(np.float32([-125.7, -126.0, -126.4, -126.6, -200.0, -1e30, -np.inf]), c)
    assert np.all(low >= 0) and np.all(low < 2.0 ** -124)
