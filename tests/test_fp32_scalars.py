"""The scalars the parity tests give the oracle.

The C ABI takes gamma, lambda, rho_bar and c_bar as fp32, so the kernel never
sees a decimal such as 0.997, only its nearest fp32 value. The parity tests
give the float64 oracle that same value (tests.parity_common.f32). These
checks run on the CPU: the rounding is the one the binding's ctypes c_float
arguments apply, and on the long-row workload the rounding alone moves the
exact discounted returns by more than the parity bar, so comparing against
the decimal would measure the input's representation, not the kernel.
"""
import ctypes

import numpy as np
import pytest

from synthetic_rollouts import WORKLOADS, workload_inputs
from tests.parity_common import TOL, f32, oracle_f32

import oracle


@pytest.mark.parametrize("x", [0.99, 0.95, 0.997, 0.999, 1.0, 0.9, 0.8, 0.5, 1e30, -2.5])
def test_f32_is_the_c_float_rounding(x):
    assert f32(x) == ctypes.c_float(x).value
    assert f32(f32(x)) == f32(x)


def test_wrapper_rounds_float_scalars_only():
    src = workload_inputs(WORKLOADS["gae_64x512"], N=4, T=64)
    args = (src["rewards"], src["values"], src["terminateds"])
    want = oracle.gae(*args, f32(0.99), f32(0.95), src["bootstrap_value"])
    got = oracle_f32.gae(*args, 0.99, lambda_=0.95, bootstrap_value=src["bootstrap_value"])
    assert np.array_equal(got, want)
    # array arguments are not scalars: they reach the oracle as given
    assert oracle_f32.affine_scan(np.full((1, 3), 0.5), np.ones((1, 3)), None, None,
                                  reverse=False).tolist() == [[1.0, 1.5, 1.75]]


def test_gamma_representation_alone_exceeds_the_bar_on_long_rows():
    w = WORKLOADS["longT_256x16384"]
    src = workload_inputs(w)
    r, d, B = src["rewards"], src["terminateds"], src["bootstrap_value"]
    exact = oracle.discounted_returns(r, d, w.gamma, B)
    at_f32 = oracle.discounted_returns(r, d, f32(w.gamma), B)
    moved = np.abs(at_f32 - exact) / np.maximum(1.0, np.abs(exact))
    assert f32(w.gamma) != w.gamma
    assert moved.max() > TOL
    # with lambda damping (GAE, lambda = 0.95) the same rounding stays far below it
    g_exact = oracle.gae(r, src["values"], d, w.gamma, w.lambda_, B)
    g_f32 = oracle.gae(r, src["values"], d, f32(w.gamma), f32(w.lambda_), B)
    assert (np.abs(g_f32 - g_exact) / np.maximum(1.0, np.abs(g_exact))).max() < TOL / 10
