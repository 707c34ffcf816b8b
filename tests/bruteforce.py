"""Explicit-sum (O(T^2)) definitions of the seven estimators, pure Python.

These are the closed sum forms of each estimator, NOT the recursions the
oracle evaluates, so agreement between the two pins the oracle to a second,
independent statement of the definition:

  * GAE as the exponentially weighted sum of TD errors (Schulman et al. 2016,
    eq. 16), stopped at the first cut.
  * Discounted returns as the truncated reward sum plus the discounted
    successor value at the first cut.
  * TD(lambda) as the lambda-weighted mixture of n-step returns, with the
    remaining weight on the complete return (Sutton & Barto, episodic
    lambda-return).
  * V-trace as IMPALA's eq. 1 sum with the products of trace weights c_i.
  * Retrace as Q(s_t, a_t) plus the sum of discounted, trace-weighted
    expected-SARSA TD errors (Munos et al. 2016).
  * Eligibility traces and the episodic prefix sum as sums from the start of
    the current episode.

Boundary conventions are the ones the page sets out under "Explicit Boundary
Semantics": a terminated step's successor value is 0, a truncated step's is
next_values[t], and the last step of the window (t = T-1) takes the bootstrap
value; a cut is any of the three. Masks count as set when nonzero.

Inputs are Python lists (one row); gamma, lambda etc. are Python numbers, so
with integer inputs and dyadic gamma/lambda every sum is exact.
"""
import math


def _cut(term, trunc, t, T):
    return term[t] != 0 or (trunc is not None and trunc[t] != 0) or t == T - 1


def _succ(values, term, trunc, nv, boot, t, T):
    if term[t] != 0:
        return 0
    if trunc is not None and trunc[t] != 0:
        return nv[t]
    if t == T - 1:
        return boot
    return values[t + 1]


def _first_cut(term, trunc, t, T):
    e = t
    while not _cut(term, trunc, e, T):
        e += 1
    return e


def gae(r, v, term, gamma, lam, boot=0, trunc=None, nv=None):
    T = len(r)
    out = []
    for t in range(T):
        e = _first_cut(term, trunc, t, T)
        total = 0
        for k in range(t, e + 1):
            nxt = v[k + 1] if k < e else _succ(v, term, trunc, nv, boot, e, T)
            delta = r[k] + gamma * nxt - v[k]
            total += (gamma * lam) ** (k - t) * delta
        out.append(total)
    return out


def discounted_returns(r, term, gamma, boot=0, trunc=None, nv=None):
    T = len(r)
    out = []
    for t in range(T):
        e = _first_cut(term, trunc, t, T)
        total = sum(gamma ** (k - t) * r[k] for k in range(t, e + 1))
        total += gamma ** (e - t + 1) * _succ(None, term, trunc, nv, boot, e, T)
        out.append(total)
    return out


def lambda_returns(r, v, term, gamma, lam, boot=0, trunc=None, nv=None):
    T = len(r)
    out = []
    for t in range(T):
        e = _first_cut(term, trunc, t, T)
        H = e - t + 1            # steps up to and including the cut

        def nstep(n):
            # n-step return G^(n)_t; n >= H is the complete return.
            m = min(n, H)
            g = sum(gamma ** k * r[t + k] for k in range(m))
            if n < H:
                g += gamma ** n * v[t + n]
            else:
                g += gamma ** H * _succ(v, term, trunc, nv, boot, e, T)
            return g

        total = (1 - lam) * sum(lam ** (n - 1) * nstep(n) for n in range(1, H))
        total += lam ** (H - 1) * nstep(H)
        out.append(total)
    return out


def vtrace(r, v, log_rho, term, gamma, lam, rho_bar, c_bar, boot=0,
           trunc=None, nv=None):
    """Returns (vs, pg_adv)."""
    T = len(r)
    ratio = [math.exp(x) for x in log_rho]
    rho = [min(rho_bar, x) for x in ratio]
    c = [lam * min(c_bar, x) for x in ratio]
    vs = []
    for t in range(T):
        e = _first_cut(term, trunc, t, T)
        total = v[t]
        for k in range(t, e + 1):
            nxt = v[k + 1] if k < e else _succ(v, term, trunc, nv, boot, e, T)
            delta = rho[k] * (r[k] + gamma * nxt - v[k])
            prod = 1
            for i in range(t, k):
                prod *= c[i]
            total += gamma ** (k - t) * prod * delta
        vs.append(total)
    pg = []
    for t in range(T):
        w = (_succ(v, term, trunc, nv, boot, t, T) if _cut(term, trunc, t, T)
             else vs[t + 1])
        pg.append(rho[t] * (r[t] + gamma * w - v[t]))
    return vs, pg


def retrace(r, v, q, log_rho, term, gamma, lam, c_bar, boot=0, trunc=None,
            nv=None):
    T = len(r)
    c = [lam * min(c_bar, math.exp(x)) for x in log_rho]
    out = []
    for t in range(T):
        e = _first_cut(term, trunc, t, T)
        total = q[t]
        for s in range(t, e + 1):
            nxt = v[s + 1] if s < e else _succ(v, term, trunc, nv, boot, e, T)
            td = r[s] + gamma * nxt - q[s]
            prod = 1
            for i in range(t + 1, s + 1):
                prod *= c[i]
            total += gamma ** (s - t) * prod * td
        out.append(total)
    return out


def _episode_start(dones, t):
    s = t
    while s > 0 and dones[s - 1] == 0:
        s -= 1
    return s


def eligibility_traces(x, dones, gamma, lam):
    out = []
    for t in range(len(x)):
        s = _episode_start(dones, t)
        out.append(sum((gamma * lam) ** (t - k) * x[k] for k in range(s, t + 1)))
    return out


def episodic_prefix_sum(x, dones):
    """Exact integer sums, wrapped to int32 like two's-complement addition."""
    out = []
    for t in range(len(x)):
        s = _episode_start(dones, t)
        total = sum(int(x[k]) for k in range(s, t + 1))
        total = (total + 2 ** 31) % 2 ** 32 - 2 ** 31
        out.append(total)
    return out


def affine_scan(a, b, reset=None, x0=0, reverse=False):
    """Explicit form: x_t = sum over k in the segment up to t of
    (product of a_j for j in (k, t]) * b_k, plus the product of every a in
    the segment times x0 when the segment reaches the origin."""
    T = len(a)
    order = list(range(T - 1, -1, -1)) if reverse else list(range(T))
    pos = {t: i for i, t in enumerate(order)}   # position along the scan
    out = [0] * T
    for t in range(T):
        total = 0
        i = pos[t]
        k = i
        while True:
            tk = order[k]
            prod = 1
            for m in range(k + 1, i + 1):
                prod *= a[order[m]]
            total += prod * b[tk]
            if reset is not None and reset[tk] != 0:
                break
            if k == 0:
                prod0 = 1
                for m in range(0, i + 1):
                    prod0 *= a[order[m]]
                total += prod0 * x0
                break
            k -= 1
        out[t] = total
    return out
