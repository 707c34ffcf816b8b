"""The scalars gamma, lambda, rho_bar and c_bar cross the C ABI as double.

Why (CPU checks on the oracle alone): rounding gamma = 0.997 to fp32 moves
it by 2.1e-8, and over the 16384-step rows of the long-row workload, where
discounted returns have no lambda damping, that alone moves the exact
returns by more than the parity bar. So the library takes the scalars in
double, computes each step in fp32, and raises the multiplier's powers that
span many steps (beta^4, beta^8, beta^16) in double before rounding them
once. The oracle is then given exactly the values the ABI receives.
"""
import ctypes

import numpy as np
import pytest

import oracle
from synthetic_rollouts import WORKLOADS, workload_inputs
from tests.parity_common import TOL


def test_rounding_gamma_to_fp32_alone_exceeds_the_bar_on_long_rows():
    w = WORKLOADS["longT_256x16384"]
    src = workload_inputs(w)
    r, d, B = src["rewards"], src["terminateds"], src["bootstrap_value"]
    g32 = float(np.float32(w.gamma))
    assert g32 != w.gamma
    exact = oracle.discounted_returns(r, d, w.gamma, B)
    moved = np.abs(oracle.discounted_returns(r, d, g32, B) - exact) / np.maximum(1.0,
                                                                                 np.abs(exact))
    assert moved.max() > TOL
    # with lambda damping (GAE, lambda = 0.95) the same rounding stays far below it
    g_exact = oracle.gae(r, src["values"], d, w.gamma, w.lambda_, B)
    g_f32 = oracle.gae(r, src["values"], d, g32, float(np.float32(w.lambda_)), B)
    assert (np.abs(g_f32 - g_exact) / np.maximum(1.0, np.abs(g_exact))).max() < TOL / 10


def test_binding_passes_the_scalars_as_double():
    rl = pytest.importorskip("linear_recurrence_scan_affine_gb300")
    lib = rl.lib()
    # rlcs_gae(r, v, d, tau, nv, boot, out, N, T, gamma, lambda, ws, ws_bytes, stream)
    assert lib.rlcs_gae.argtypes[9:11] == [ctypes.c_double, ctypes.c_double]
    # rlcs_vtrace(..., N, T, gamma, lambda, rho_bar, c_bar, ws, ws_bytes, stream)
    assert lib.rlcs_vtrace.argtypes[11:15] == [ctypes.c_double] * 4
    from linear_recurrence_scan_affine_gb300.binding import RlcsCall
    assert all(t is ctypes.c_double for f, t in RlcsCall._fields_
               if f in ("gamma", "lambda_", "rho_bar", "c_bar"))


def test_header_declares_no_fp32_scalars():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "rlcs.h")).read()
    assert not re.search(r"\bfloat\s+(gamma|lambda|rho_bar|c_bar)\b", hdr)
    assert re.search(r"\bdouble\s+gamma\b", hdr)
