"""Float64 CPU oracle for the seven credit-assignment estimators.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package; the product path never does.
It shares no code with the CUDA library. The arithmetic lives in
``rlcs_oracle.c`` (each function there cites the page passage it follows);
this module only loads it and marshals numpy arrays.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        # RLCS_ORACLE_LIB lets the mutation tests point the pins at a
        # deliberately broken build of this oracle.
        path = os.environ.get("RLCS_ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        i64, dbl, ptr = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_gae.argtypes = [i64, i64] + [ptr] * 6 + [dbl, dbl, ptr]
        lib.oracle_lambda_returns.argtypes = [i64, i64] + [ptr] * 6 + [dbl, dbl, ptr]
        lib.oracle_discounted_returns.argtypes = [i64, i64] + [ptr] * 5 + [dbl, ptr]
        lib.oracle_vtrace.argtypes = [i64, i64] + [ptr] * 7 + [dbl] * 4 + [ptr, ptr]
        lib.oracle_retrace.argtypes = [i64, i64] + [ptr] * 8 + [dbl] * 3 + [ptr]
        lib.oracle_eligibility_traces.argtypes = [i64, i64, ptr, ptr, dbl, dbl, ptr]
        lib.oracle_episodic_prefix_sum.argtypes = [i64, i64, ptr, ptr, ptr]
        lib.oracle_affine_scan.argtypes = [i64, i64, ptr, ptr, ptr, ptr, ctypes.c_int, ptr]
        for f in (lib.oracle_gae, lib.oracle_lambda_returns,
                  lib.oracle_discounted_returns, lib.oracle_vtrace,
                  lib.oracle_retrace, lib.oracle_eligibility_traces,
                  lib.oracle_episodic_prefix_sum, lib.oracle_affine_scan):
            f.restype = None
        _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shape(a):
    a = np.asarray(a)
    if a.ndim == 1:
        return 1, a.shape[0]
    assert a.ndim == 2
    return a.shape


def _trunc(truncateds, next_values):
    if (truncateds is None) != (next_values is None):
        raise ValueError("truncateds and next_values go together")
    return _f32(truncateds), _f32(next_values)


def _boot(bootstrap_value, N):
    if bootstrap_value is None:
        return None
    b = _f32(bootstrap_value).reshape(-1)
    assert b.shape[0] == N
    return b


def gae(rewards, values, terminateds, gamma, lambda_, bootstrap_value=None,
        truncateds=None, next_values=None):
    N, T = _shape(rewards)
    r, v, d = _f32(rewards), _f32(values), _f32(terminateds)
    tr, nv = _trunc(truncateds, next_values)
    b = _boot(bootstrap_value, N)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_gae(N, T, _p(r), _p(v), _p(d), _p(tr), _p(nv), _p(b),
                       gamma, lambda_, _p(out))
    return out.reshape(np.shape(rewards))


def lambda_returns(rewards, values, terminateds, gamma, lambda_,
                   bootstrap_value=None, truncateds=None, next_values=None):
    N, T = _shape(rewards)
    r, v, d = _f32(rewards), _f32(values), _f32(terminateds)
    tr, nv = _trunc(truncateds, next_values)
    b = _boot(bootstrap_value, N)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_lambda_returns(N, T, _p(r), _p(v), _p(d), _p(tr), _p(nv),
                                  _p(b), gamma, lambda_, _p(out))
    return out.reshape(np.shape(rewards))


def discounted_returns(rewards, terminateds, gamma, bootstrap_value=None,
                       truncateds=None, next_values=None):
    N, T = _shape(rewards)
    r, d = _f32(rewards), _f32(terminateds)
    tr, nv = _trunc(truncateds, next_values)
    b = _boot(bootstrap_value, N)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_discounted_returns(N, T, _p(r), _p(d), _p(tr), _p(nv),
                                      _p(b), gamma, _p(out))
    return out.reshape(np.shape(rewards))


def vtrace(rewards, values, log_rhos, terminateds, gamma, lambda_, rho_bar,
           c_bar, bootstrap_value=None, truncateds=None, next_values=None):
    """Returns (vs, pg_advantages), both float64."""
    N, T = _shape(rewards)
    r, v, lr, d = _f32(rewards), _f32(values), _f32(log_rhos), _f32(terminateds)
    tr, nv = _trunc(truncateds, next_values)
    b = _boot(bootstrap_value, N)
    vs = np.empty((N, T), dtype=np.float64)
    pg = np.empty((N, T), dtype=np.float64)
    _load().oracle_vtrace(N, T, _p(r), _p(v), _p(lr), _p(d), _p(tr), _p(nv),
                          _p(b), gamma, lambda_, rho_bar, c_bar, _p(vs), _p(pg))
    shp = np.shape(rewards)
    return vs.reshape(shp), pg.reshape(shp)


def retrace(rewards, values, q_values, log_rhos, terminateds, gamma, lambda_,
            c_bar, bootstrap_value=None, truncateds=None, next_values=None):
    N, T = _shape(rewards)
    r, v, q = _f32(rewards), _f32(values), _f32(q_values)
    lr, d = _f32(log_rhos), _f32(terminateds)
    tr, nv = _trunc(truncateds, next_values)
    b = _boot(bootstrap_value, N)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_retrace(N, T, _p(r), _p(v), _p(q), _p(lr), _p(d), _p(tr),
                           _p(nv), _p(b), gamma, lambda_, c_bar, _p(out))
    return out.reshape(np.shape(rewards))


def eligibility_traces(x, dones, gamma, lambda_):
    N, T = _shape(x)
    xx, d = _f32(x), _f32(dones)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_eligibility_traces(N, T, _p(xx), _p(d), gamma, lambda_,
                                      _p(out))
    return out.reshape(np.shape(x))


def episodic_prefix_sum(x, dones):
    N, T = _shape(x)
    xx = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    d = _f32(dones)
    out = np.empty((N, T), dtype=np.int32)
    _load().oracle_episodic_prefix_sum(N, T, _p(xx), _p(d), _p(out))
    return out.reshape(np.shape(x))


def affine_scan(a, b, reset=None, x_init=None, reverse=False):
    """x_t = a_t*x_{t-1} + b_t (or the reverse-time mirror), float64."""
    N, T = _shape(a)
    aa, bb, rr = _f32(a), _f32(b), _f32(reset)
    x0 = _boot(x_init, N)
    out = np.empty((N, T), dtype=np.float64)
    _load().oracle_affine_scan(N, T, _p(aa), _p(bb), _p(rr), _p(x0), 1 if reverse else 0,
                               _p(out))
    return out.reshape(np.shape(a))
