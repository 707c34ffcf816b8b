"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is chosen so a plausible slip in the oracle (a dropped term, a wrong
sign, an index off by one, a mask applied at the wrong step) fails at least
one test:
  * closed forms (constant reward / constant input, no dones);
  * special cases that reduce to other estimators or to textbook routines
    (lambda=0 -> one-step TD error, lambda=1 -> Monte Carlo, unit ratios ->
    on-policy, numpy.cumsum for the prefix sum);
  * the explicit-sum definitions of ``bruteforce.py`` on short rows, exhaustive
    over every done pattern at T <= 8 with exact (integer, dyadic) arithmetic;
  * structural invariants (no bleed across a terminated step, truncation =
    split rollout, time-reversal duality between traces and returns);
  * hand-derived worked examples stored under tests/golden/.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from synthetic_rollouts import rollout
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RTOL = 1e-12


def close(a, b, tol=RTOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.all(np.abs(a - b) <= tol * np.maximum(1.0, np.abs(b)))


def inputs(N, T, seed, p_term=0.1, p_trunc=0.0):
    return rollout(N, T, seed, p_term, p_trunc)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.99, 0.997])
def test_discounted_returns_closed_form(gamma):
    T, rew = 300, 0.75
    r = np.full((1, T), rew, np.float32)
    d = np.zeros((1, T), np.float32)
    g = oracle.discounted_returns(r, d, gamma)[0]
    t = np.arange(T)
    expect = rew * (1 - gamma ** (T - t)) / (1 - gamma)
    assert close(g, expect, 1e-12)


@pytest.mark.parametrize("gamma,lam", [(0.99, 0.95), (0.5, 0.5), (0.999, 1.0)])
def test_eligibility_traces_closed_form(gamma, lam):
    T, xv = 257, -1.25
    x = np.full((2, T), xv, np.float32)
    d = np.zeros((2, T), np.float32)
    e = oracle.eligibility_traces(x, d, gamma, lam)
    t = np.arange(T)
    gl = gamma * lam
    expect = xv * (1 - gl ** (t + 1)) / (1 - gl) if gl != 1 else xv * (t + 1)
    assert close(e[0], expect) and close(e[1], expect)


def test_all_done_reduces_to_one_step():
    src = inputs(3, 37, 7)
    r, v, lr, q = src["rewards"], src["values"], src["log_rhos"], src["q_values"]
    d = np.ones_like(r)
    b = src["bootstrap_value"]
    rd = r.astype(np.float64)
    assert close(oracle.gae(r, v, d, 0.99, 0.95, b), rd - v)
    assert close(oracle.lambda_returns(r, v, d, 0.99, 0.95, b), rd)
    assert close(oracle.discounted_returns(r, d, 0.99, b), rd)
    assert close(oracle.retrace(r, v, q, lr, d, 0.99, 0.95, 1.0, b), rd)
    vs, pg = oracle.vtrace(r, v, lr, d, 0.99, 0.95, 1.0, 1.0, b)
    rho = np.minimum(1.0, np.exp(lr.astype(np.float64)))
    assert close(vs, v + rho * (rd - v))
    assert close(pg, rho * (rd - v))


# --------------------------------------------------------------------------
# Special cases and cross-estimator identities
# --------------------------------------------------------------------------

@pytest.mark.parametrize("trunc", [False, True])
def test_gae_lambda0_is_td_error(trunc):
    src = inputs(4, 50, 11, p_term=0.1, p_trunc=0.08 if trunc else 0.0)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src.get("truncateds"), src.get("next_values")
    a = oracle.gae(r, v, d, 0.9, 0.0, b, tr, nv)
    # one-step TD error written from the boundary rules, column by column
    N, T = r.shape
    succ = np.zeros((N, T))
    succ[:, :-1] = v[:, 1:]
    succ[:, -1] = b
    if trunc:
        succ = np.where(tr != 0, nv, succ)
    succ = np.where(d != 0, 0.0, succ)
    assert close(a, r + 0.9 * succ - v)


@pytest.mark.parametrize("trunc", [False, True])
def test_gae_lambda1_is_monte_carlo_minus_value(trunc):
    src = inputs(4, 64, 12, p_term=0.05, p_trunc=0.05 if trunc else 0.0)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src.get("truncateds"), src.get("next_values")
    a = oracle.gae(r, v, d, 0.97, 1.0, b, tr, nv)
    g = oracle.discounted_returns(r, d, 0.97, b, tr, nv)
    assert close(a, g - v, 1e-11)


@pytest.mark.parametrize("lam", [0.0, 0.3, 0.95, 1.0])
@pytest.mark.parametrize("trunc", [False, True])
def test_lambda_returns_equal_gae_plus_value(lam, trunc):
    src = inputs(3, 80, 13, p_term=0.05, p_trunc=0.05 if trunc else 0.0)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src.get("truncateds"), src.get("next_values")
    g = oracle.lambda_returns(r, v, d, 0.99, lam, b, tr, nv)
    a = oracle.gae(r, v, d, 0.99, lam, b, tr, nv)
    assert close(g, a + v, 1e-11)


@pytest.mark.parametrize("trunc", [False, True])
def test_vtrace_on_policy_is_lambda_return(trunc):
    src = inputs(3, 90, 14, p_term=0.05, p_trunc=0.05 if trunc else 0.0)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src.get("truncateds"), src.get("next_values")
    zero = np.zeros_like(r)
    for rho_bar, c_bar in [(1.0, 1.0), (2.0, 1.5)]:
        vs, pg = oracle.vtrace(r, v, zero, d, 0.98, 0.9, rho_bar, c_bar, b, tr, nv)
        g = oracle.lambda_returns(r, v, d, 0.98, 0.9, b, tr, nv)
        assert close(vs, g, 1e-11)
        # pg advantage with unit ratios: r + gamma*W - V, W = vs_{t+1} or S_t
        delta0 = oracle.gae(r, v, d, 0.98, 0.0, b, tr, nv)   # r + gamma*S - V
        N, T = r.shape
        cut = (d != 0)
        if trunc:
            cut |= (tr != 0)
        cut[:, -1] = True
        expect = delta0.copy()
        expect[:, :-1] = np.where(cut[:, :-1], delta0[:, :-1],
                                  r[:, :-1] + 0.98 * vs[:, 1:] - v[:, :-1])
        assert close(pg, expect, 1e-11)


def test_vtrace_clipping_limits():
    src = inputs(2, 40, 15)
    r, v, lr, d, b = (src[k] for k in ("rewards", "values", "log_rhos",
                                       "terminateds", "bootstrap_value"))
    # c_bar = 0: no trace, vs = V + rho * delta
    vs, _ = oracle.vtrace(r, v, lr, d, 0.99, 0.95, 1.0, 0.0, b)
    delta = oracle.gae(r, v, d, 0.99, 0.0, b)
    rho = np.minimum(1.0, np.exp(lr.astype(np.float64)))
    assert close(vs, v + rho * delta)
    # rho_bar = 0: nothing moves, vs = V and pg = 0
    vs, pg = oracle.vtrace(r, v, lr, d, 0.99, 0.95, 0.0, 1.0, b)
    assert close(vs, v) and np.all(pg == 0)


def test_vtrace_lambda_placement():
    # lambda multiplies the trace weight c only: with rho clipped to 1 and
    # unit ratios, lambda=0 gives vs = V + delta (one-step), lambda=1 gives
    # the Monte Carlo return.
    src = inputs(2, 60, 16, p_term=0.05)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    zero = np.zeros_like(r)
    vs0, _ = oracle.vtrace(r, v, zero, d, 0.95, 0.0, 1.0, 1.0, b)
    assert close(vs0, v + oracle.gae(r, v, d, 0.95, 0.0, b))
    vs1, _ = oracle.vtrace(r, v, zero, d, 0.95, 1.0, 1.0, 1.0, b)
    assert close(vs1, oracle.discounted_returns(r, d, 0.95, b), 1e-11)


@pytest.mark.parametrize("trunc", [False, True])
def test_retrace_on_policy_is_lambda_return(trunc):
    src = inputs(3, 70, 17, p_term=0.05, p_trunc=0.05 if trunc else 0.0)
    r, v, d, b = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src.get("truncateds"), src.get("next_values")
    zero = np.zeros_like(r)
    q = oracle.retrace(r, v, v, zero, d, 0.99, 0.8, 1.0, b, tr, nv)
    g = oracle.lambda_returns(r, v, d, 0.99, 0.8, b, tr, nv)
    assert close(q, g, 1e-11)
    # lambda = 0: expected-SARSA target r + gamma*S
    q0 = oracle.retrace(r, v, src["q_values"], src["log_rhos"], d, 0.99, 0.0,
                        1.0, b, tr, nv)
    assert close(q0, oracle.gae(r, v, d, 0.99, 0.0, b, tr, nv) + v)


def test_retrace_trace_uses_next_ratio():
    # Changing log_rho at t only changes Q^ret at t-1 and earlier (the trace
    # c_{t} weighs the correction carried into step t-1), never at t itself.
    src = inputs(1, 30, 18, p_term=0.0)
    r, v, q, lr, d = (src[k] for k in ("rewards", "values", "q_values",
                                       "log_rhos", "terminateds"))
    base = oracle.retrace(r, v, q, lr, d, 0.9, 0.9, 1.0)
    lr2 = lr.copy()
    lr2[0, 20] -= 2.0
    alt = oracle.retrace(r, v, q, lr2, d, 0.9, 0.9, 1.0)
    assert np.all(alt[0, 20:] == base[0, 20:])
    assert alt[0, 19] != base[0, 19]


def test_prefix_sum_textbook_cases():
    src = inputs(3, 200, 19)
    x = src["x_int"]
    zero = np.zeros((3, 200), np.float32)
    s = oracle.episodic_prefix_sum(x, zero)
    assert np.array_equal(s, np.cumsum(x.astype(np.int64), axis=1).astype(np.int32))
    assert np.array_equal(oracle.episodic_prefix_sum(x, np.ones_like(zero)), x)


def test_prefix_sum_wraps_mod_2_32():
    x = np.array([[2 ** 31 - 1, 5, -7, 2 ** 31 - 1, 2 ** 31 - 1]], np.int32)
    d = np.zeros_like(x, dtype=np.float32)
    s = oracle.episodic_prefix_sum(x, d)
    assert s.tolist() == [bf.episodic_prefix_sum(x[0].tolist(), [0] * 5)]


def test_elig_is_time_reversed_discounted_return():
    src = inputs(3, 64, 20, p_term=0.1)
    x, d = src["x"], src["terminateds"]
    gamma, lam = 0.97, 0.8
    e = oracle.eligibility_traces(x, d, gamma, lam)
    xr = x[:, ::-1]
    dr = np.ones_like(d)
    dr[:, :-1] = d[:, :-1][:, ::-1]       # d'_u = d_{T-2-u}, u <= T-2
    g = oracle.discounted_returns(xr, dr, gamma * lam)
    assert close(e, g[:, ::-1], 1e-11)


# --------------------------------------------------------------------------
# Boundary structure
# --------------------------------------------------------------------------

def _backward_all(src, gamma=0.99, lam=0.95, trunc=True):
    r, v, q, lr, d, b = (src[k] for k in ("rewards", "values", "q_values",
                                          "log_rhos", "terminateds",
                                          "bootstrap_value"))
    tr, nv = (src.get("truncateds"), src.get("next_values")) if trunc else (None, None)
    vs, pg = oracle.vtrace(r, v, lr, d, gamma, lam, 1.0, 1.0, b, tr, nv)
    return {
        "gae": oracle.gae(r, v, d, gamma, lam, b, tr, nv),
        "lret": oracle.lambda_returns(r, v, d, gamma, lam, b, tr, nv),
        "disc": oracle.discounted_returns(r, d, gamma, b, tr, nv),
        "vs": vs, "pg": pg,
        "retrace": oracle.retrace(r, v, q, lr, d, gamma, lam, 1.0, b, tr, nv),
    }


def test_no_bleed_across_terminated_step():
    T, td = 40, 17
    src = inputs(1, T, 21, p_term=0.0, p_trunc=0.05)
    src["terminateds"][0, td] = 1.0
    src["truncateds"][0, td] = 0.0
    base = _backward_all(src)
    pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in src.items()}
    rng = np.random.default_rng(0)
    for k in ("rewards", "values", "q_values", "log_rhos", "next_values"):
        pert[k][0, td + 1:] += rng.standard_normal(T - td - 1).astype(np.float32)
    pert["bootstrap_value"] = pert["bootstrap_value"] + 3.0
    alt = _backward_all(pert)
    for k in base:
        assert np.array_equal(base[k][0, :td + 1], alt[k][0, :td + 1]), k
        assert not np.array_equal(base[k][0, td + 1:], alt[k][0, td + 1:]), k
    # forward estimators: a done at td shields t > td from inputs at <= td
    x, xi, d = src["x"], src["x_int"], src["terminateds"]
    e0 = oracle.eligibility_traces(x, d, 0.9, 0.9)
    s0 = oracle.episodic_prefix_sum(xi, d)
    x2, xi2 = x.copy(), xi.copy()
    x2[0, :td + 1] += 1.0
    xi2[0, :td + 1] += 3
    e1 = oracle.eligibility_traces(x2, d, 0.9, 0.9)
    s1 = oracle.episodic_prefix_sum(xi2, d)
    assert np.array_equal(e0[0, td + 1:], e1[0, td + 1:])
    assert np.array_equal(s0[0, td + 1:], s1[0, td + 1:])
    assert not np.array_equal(e0[0, :td + 1], e1[0, :td + 1])


@pytest.mark.parametrize("kind", ["truncated", "terminated"])
def test_boundary_step_equals_split_rollout(kind):
    T, ts = 33, 12
    src = inputs(1, T, 22, p_term=0.0, p_trunc=0.0)
    src["truncateds"] = np.zeros((1, T), np.float32)
    src["next_values"] = rollout(1, T, 99, 0.0)["values"]
    whole = dict(src)
    if kind == "truncated":
        whole["truncateds"] = src["truncateds"].copy()
        whole["truncateds"][0, ts] = 1.0
        split_boot = src["next_values"][0, ts]
    else:
        whole["terminateds"] = src["terminateds"].copy()
        whole["terminateds"][0, ts] = 1.0
        split_boot = 0.0
    ref = _backward_all(whole)
    first = {k: (v[:, :ts + 1] if isinstance(v, np.ndarray) and v.ndim == 2 else v)
             for k, v in src.items()}
    first["bootstrap_value"] = np.array([split_boot], np.float32)
    second = {k: (v[:, ts + 1:] if isinstance(v, np.ndarray) and v.ndim == 2 else v)
              for k, v in src.items()}
    a, b = _backward_all(first), _backward_all(second)
    for k in ref:
        assert close(ref[k][0, :ts + 1], a[k][0], 1e-14), k
        assert close(ref[k][0, ts + 1:], b[k][0], 1e-14), k


# --------------------------------------------------------------------------
# Brute force: explicit-sum definitions
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 2, 3, 5, 8, 13, 16])
@pytest.mark.parametrize("trunc", [False, True])
def test_bruteforce_random(T, trunc):
    src = inputs(6, T, 100 + T, p_term=0.2, p_trunc=0.15 if trunc else 0.0)
    gamma, lam, rho_bar, c_bar = 0.93, 0.71, 1.1, 0.9
    r, v, q, lr, d, b = (src[k] for k in ("rewards", "values", "q_values",
                                          "log_rhos", "terminateds",
                                          "bootstrap_value"))
    tr, nv = src.get("truncateds"), src.get("next_values")
    o = {
        "gae": oracle.gae(r, v, d, gamma, lam, b, tr, nv),
        "lret": oracle.lambda_returns(r, v, d, gamma, lam, b, tr, nv),
        "disc": oracle.discounted_returns(r, d, gamma, b, tr, nv),
        "vt": oracle.vtrace(r, v, lr, d, gamma, lam, rho_bar, c_bar, b, tr, nv),
        "ret": oracle.retrace(r, v, q, lr, d, gamma, lam, c_bar, b, tr, nv),
        "elig": oracle.eligibility_traces(src["x"], d, gamma, lam),
        "psum": oracle.episodic_prefix_sum(src["x_int"], d),
    }
    for n in range(6):
        L = lambda a: [float(z) for z in a[n]]
        kw = dict(boot=float(b[n]))
        if trunc:
            kw.update(trunc=L(tr), nv=L(nv))
        assert close(o["gae"][n], bf.gae(L(r), L(v), L(d), gamma, lam, **kw))
        assert close(o["lret"][n], bf.lambda_returns(L(r), L(v), L(d), gamma, lam, **kw))
        assert close(o["disc"][n], bf.discounted_returns(L(r), L(d), gamma, **kw))
        vs, pg = bf.vtrace(L(r), L(v), L(lr), L(d), gamma, lam, rho_bar, c_bar, **kw)
        assert close(o["vt"][0][n], vs) and close(o["vt"][1][n], pg)
        assert close(o["ret"][n], bf.retrace(L(r), L(v), L(q), L(lr), L(d), gamma,
                                             lam, c_bar, **kw))
        assert close(o["elig"][n], bf.eligibility_traces(L(src["x"]), L(d), gamma, lam))
        assert o["psum"][n].tolist() == bf.episodic_prefix_sum(
            src["x_int"][n].tolist(), L(d))


@pytest.mark.parametrize("T,both", [(1, False), (4, False), (7, False), (2, True), (5, True)])
def test_bruteforce_exhaustive_exact(T, both):
    """Every (terminated, truncated) pattern with small integer inputs and
    dyadic gamma/lambda: the oracle and the explicit sums must agree exactly.
    With `both`, steps may also carry both masks at once (termination wins)."""
    rng = np.random.default_rng(T)
    gamma, lam = 0.5, 0.75
    r = rng.integers(-4, 5, T).astype(np.float32)
    v = rng.integers(-4, 5, T).astype(np.float32)
    q = rng.integers(-4, 5, T).astype(np.float32)
    nv = rng.integers(-4, 5, T).astype(np.float32)
    x = rng.integers(-4, 5, T).astype(np.float32)
    xi = rng.integers(-100, 101, T).astype(np.int32)
    zero = np.zeros(T, np.float32)
    boot = 3.0
    kinds = [0, 1, 2, 3] if both else [0, 1, 2]  # none, term, trunc, both
    pats = list(itertools.product(kinds, repeat=T))
    for pat in pats:
        d = np.array([p in (1, 3) for p in pat], np.float32)
        tr = np.array([p in (2, 3) for p in pat], np.float32)
        kw = dict(boot=boot, trunc=tr.tolist(), nv=nv.tolist())
        B = np.array([boot], np.float32)
        got = oracle.gae(r[None], v[None], d[None], gamma, lam, B, tr[None], nv[None])[0]
        assert got.tolist() == bf.gae(r.tolist(), v.tolist(), d.tolist(), gamma, lam, **kw)
        got = oracle.lambda_returns(r[None], v[None], d[None], gamma, lam, B,
                                    tr[None], nv[None])[0]
        assert got.tolist() == bf.lambda_returns(r.tolist(), v.tolist(), d.tolist(),
                                                 gamma, lam, **kw)
        got = oracle.discounted_returns(r[None], d[None], gamma, B, tr[None], nv[None])[0]
        assert got.tolist() == bf.discounted_returns(r.tolist(), d.tolist(), gamma, **kw)
        # unit ratios keep V-trace and Retrace exact (exp(0) = 1)
        vs, pg = oracle.vtrace(r[None], v[None], zero[None], d[None], gamma, lam,
                               1.0, 1.0, B, tr[None], nv[None])
        bvs, bpg = bf.vtrace(r.tolist(), v.tolist(), zero.tolist(), d.tolist(),
                             gamma, lam, 1.0, 1.0, **kw)
        assert vs[0].tolist() == bvs and pg[0].tolist() == bpg
        got = oracle.retrace(r[None], v[None], q[None], zero[None], d[None], gamma,
                             lam, 1.0, B, tr[None], nv[None])[0]
        assert got.tolist() == bf.retrace(r.tolist(), v.tolist(), q.tolist(),
                                          zero.tolist(), d.tolist(), gamma, lam, 1.0, **kw)
        dd = np.array([p != 0 for p in pat], np.float32)
        got = oracle.eligibility_traces(x[None], dd[None], gamma, lam)[0]
        assert got.tolist() == bf.eligibility_traces(x.tolist(), dd.tolist(), gamma, lam)
        got = oracle.episodic_prefix_sum(xi[None], dd[None])[0]
        assert got.tolist() == bf.episodic_prefix_sum(xi.tolist(), dd.tolist())


# --------------------------------------------------------------------------
# The affine operator (Methodology 1)
# --------------------------------------------------------------------------

def _op(earlier, later):
    """(alpha_B, beta_B) (+) (alpha_A, beta_A) = (alpha_B + beta_B*alpha_A,
    beta_A*beta_B), B the step nearer the output's time origin."""
    (ab, bb), (aa, ba) = earlier, later
    return (ab + bb * aa, ba * bb)


def test_operator_associative_exact():
    rng = np.random.default_rng(5)
    for _ in range(2000):
        x, y, z = [(int(a), int(b)) for a, b in rng.integers(-50, 51, (3, 2))]
        assert _op(_op(x, y), z) == _op(x, _op(y, z))


def test_operator_scan_reproduces_recursion():
    """Folding the operator over per-step (alpha, beta) pairs of GAE gives the
    recursion's result at every t, for any bracketing (checked with a random
    balanced tree and a right fold), exact with dyadic numbers."""
    from fractions import Fraction as F
    rng = np.random.default_rng(6)
    T = 12
    gamma, lam = F(1, 2), F(3, 4)
    r = [int(z) for z in rng.integers(-5, 6, T)]
    v = [int(z) for z in rng.integers(-5, 6, T)]
    d = [int(z) for z in (rng.random(T) < 0.25)]
    boot = 2
    pairs = []
    for t in range(T):
        cut = d[t] or t == T - 1
        s = 0 if d[t] else (boot if t == T - 1 else v[t + 1])
        pairs.append((r[t] + gamma * s - v[t], 0 if cut else gamma * lam))
    ref = oracle.gae(np.array([r], np.float32), np.array([v], np.float32),
                     np.array([d], np.float32), 0.5, 0.75,
                     np.array([boot], np.float32))[0]

    def tree(ps):
        if len(ps) == 1:
            return ps[0]
        k = int(rng.integers(1, len(ps)))
        return _op(tree(ps[:k]), tree(ps[k:]))

    for t in range(T):
        a_tree = tree(pairs[t:])[0]
        a_fold = pairs[-1]
        for p in reversed(pairs[t:-1]):
            a_fold = _op(p, a_fold)
        assert float(a_tree) == ref[t] == float(a_fold[0])


# --------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden)
# --------------------------------------------------------------------------

def _golden_cases():
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json"))


@pytest.mark.parametrize("fname", _golden_cases())
def test_golden_worked_examples(fname):
    with open(os.path.join(GOLDEN, fname)) as fh:
        case = json.load(fh)
    a = {k: np.array([v], dtype=np.int32 if k == "x_int" else np.float32)
         for k, v in case["inputs"].items()}
    p = case["params"]
    B = np.array([p.get("bootstrap", 0.0)], np.float32)
    tr, nv = a.get("truncateds"), a.get("next_values")
    est = case["estimator"]
    if est == "gae":
        got = {"out": oracle.gae(a["rewards"], a["values"], a["terminateds"],
                                 p["gamma"], p["lambda"], B, tr, nv)}
    elif est == "lambda_returns":
        got = {"out": oracle.lambda_returns(a["rewards"], a["values"],
                                            a["terminateds"], p["gamma"],
                                            p["lambda"], B, tr, nv)}
    elif est == "discounted_returns":
        got = {"out": oracle.discounted_returns(a["rewards"], a["terminateds"],
                                                p["gamma"], B, tr, nv)}
    elif est == "vtrace":
        vs, pg = oracle.vtrace(a["rewards"], a["values"], a["log_rhos"],
                               a["terminateds"], p["gamma"], p["lambda"],
                               p["rho_bar"], p["c_bar"], B, tr, nv)
        got = {"vs": vs, "pg": pg}
    elif est == "retrace":
        got = {"out": oracle.retrace(a["rewards"], a["values"], a["q_values"],
                                     a["log_rhos"], a["terminateds"],
                                     p["gamma"], p["lambda"], p["c_bar"], B,
                                     tr, nv)}
    elif est == "eligibility_traces":
        got = {"out": oracle.eligibility_traces(a["x"], a["dones"], p["gamma"],
                                                p["lambda"])}
    elif est == "episodic_prefix_sum":
        got = {"out": oracle.episodic_prefix_sum(a["x_int"], a["dones"])}
    else:
        raise AssertionError(est)
    for k, want in case["expected"].items():
        assert close(got[k][0], want, 1e-12), (fname, k, got[k][0], want)


# --------------------------------------------------------------------------
# Generic affine scan (the recurrence itself, on raw coefficients)
# --------------------------------------------------------------------------

def test_affine_closed_form():
    T, av, bv, x0 = 200, 0.97, 0.5, 3.0
    a = np.full((1, T), av, np.float32)
    b = np.full((1, T), bv, np.float32)
    x = oracle.affine_scan(a, b, x_init=np.array([x0], np.float32))[0]
    t = np.arange(T)
    af = float(np.float32(av))
    expect = af ** (t + 1) * x0 + bv * (1 - af ** (t + 1)) / (1 - af)
    assert close(x, expect, 1e-12)


def test_affine_reverse_is_mirrored_forward():
    rng = np.random.default_rng(30)
    a = rng.uniform(-1, 1, (3, 90)).astype(np.float32)
    b = rng.standard_normal((3, 90)).astype(np.float32)
    r = (rng.random((3, 90)) < 0.05).astype(np.float32)
    x0 = rng.standard_normal(3).astype(np.float32)
    fwd = oracle.affine_scan(a[:, ::-1], b[:, ::-1], r[:, ::-1], x0)
    rev = oracle.affine_scan(a, b, r, x0, reverse=True)
    assert np.array_equal(rev, fwd[:, ::-1])


def test_affine_reset_everywhere_is_b():
    rng = np.random.default_rng(31)
    a = rng.standard_normal((2, 40)).astype(np.float32)
    b = rng.standard_normal((2, 40)).astype(np.float32)
    for rev in (False, True):
        x = oracle.affine_scan(a, b, np.ones_like(a), np.ones(2, np.float32), reverse=rev)
        assert np.array_equal(x, b.astype(np.float64))


def test_affine_reproduces_gae_and_traces():
    """The estimators are instances of the recurrence (Methodology 1): GAE's
    coefficients in the reverse scan give the pinned GAE oracle; the traces'
    coefficients in the forward scan give the pinned traces oracle."""
    src = inputs(4, 70, 32, p_term=0.05, p_trunc=0.05)
    r, v, d, B = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    tr, nv = src["truncateds"], src["next_values"]
    g, lam = 0.5, 0.75                      # dyadic: the coefficients are exact
    delta = oracle.gae(r, v, d, g, 0.0, B, tr, nv)        # = r + g*S - V
    cut = (d != 0) | (tr != 0)
    cut[:, -1] = True
    a = np.where(cut, 0.0, g * lam).astype(np.float32)
    want = oracle.gae(r, v, d, g, lam, B, tr, nv)
    got = oracle.affine_scan(a, delta.astype(np.float32), reverse=True)
    # delta was rounded to fp32 to feed the scan: compare at fp32 precision
    assert close(got, want, 1e-6)
    x = src["x"]
    a2 = np.zeros_like(x)
    a2[:, 1:] = np.where(d[:, :-1] != 0, 0.0, g * lam)
    assert np.array_equal(oracle.affine_scan(a2, x), oracle.eligibility_traces(x, d, g, lam))


@pytest.mark.parametrize("T", [1, 2, 5])
def test_affine_bruteforce_exhaustive(T):
    rng = np.random.default_rng(33 + T)
    a = (rng.integers(-4, 5, T) / 4).astype(np.float32)
    b = rng.integers(-4, 5, T).astype(np.float32)
    for pat in itertools.product([0, 1], repeat=T):
        rs = np.array(pat, np.float32)
        for rev in (False, True):
            got = oracle.affine_scan(a[None], b[None], rs[None], np.array([2.0], np.float32),
                                     reverse=rev)[0]
            want = bf.affine_scan(a.tolist(), b.tolist(), rs.tolist(), 2.0, rev)
            assert got.tolist() == want
