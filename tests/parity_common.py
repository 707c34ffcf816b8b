"""Shared helpers for the GPU parity tests: run every estimator through the
CUDA library and through the float64 oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle

TOL = 1e-4          # |gpu - oracle| <= TOL * max(1, |oracle|) for T <= 16384
TOL_VLONG = 1e-3    # same bound at T = 131072


BACKWARD = ("gae", "lambda_returns", "discounted_returns", "vtrace", "retrace")
FORWARD = ("eligibility_traces", "episodic_prefix_sum")
ALL = BACKWARD + FORWARD


def to_dev(src, dev, offset=0):
    """Copy numpy inputs to the device. offset > 0 places every [N, T] array
    `offset` elements into a larger buffer so rows lose 16-byte alignment."""
    out = {}
    for k, v in src.items():
        t = torch.from_numpy(np.ascontiguousarray(v))
        if offset and v.ndim == 2:
            flat = torch.empty(v.size + offset, dtype=t.dtype, device=dev)
            flat[offset:] = t.reshape(-1).to(dev)
            out[k] = flat[offset:].view(v.shape)
        else:
            out[k] = t.to(dev)
    return out


def run_gpu(rl, est, g, prm, trunc):
    tr = dict(truncateds=g["truncateds"], next_values=g["next_values"]) if trunc else {}
    B = g.get("bootstrap_value")
    gm, lm = prm["gamma"], prm["lambda_"]
    if est == "gae":
        return {"out": rl.rlcs_gae(g["rewards"], g["values"], g["terminateds"], gm, lm, B, **tr)}
    if est == "lambda_returns":
        return {"out": rl.rlcs_lambda_returns(g["rewards"], g["values"], g["terminateds"], gm, lm,
                                              B, **tr)}
    if est == "discounted_returns":
        return {"out": rl.rlcs_discounted_returns(g["rewards"], g["terminateds"], gm, B, **tr)}
    if est == "vtrace":
        vs, pg = rl.rlcs_vtrace(g["rewards"], g["values"], g["log_rhos"], g["terminateds"], gm,
                                lm, prm["rho_bar"], prm["c_bar"], B, **tr)
        return {"vs": vs, "pg": pg}
    if est == "retrace":
        return {"out": rl.rlcs_retrace(g["rewards"], g["values"], g["q_values"], g["log_rhos"],
                                       g["terminateds"], gm, lm, prm["c_bar"], B, **tr)}
    if est == "eligibility_traces":
        return {"out": rl.rlcs_eligibility_traces(g["x"], g["terminateds"], gm, lm)}
    if est == "episodic_prefix_sum":
        return {"out": rl.rlcs_episodic_prefix_sum(g["x_int"], g["terminateds"])}
    raise ValueError(est)


def run_oracle(est, src, prm, trunc):
    tr = dict(truncateds=src["truncateds"], next_values=src["next_values"]) if trunc else {}
    B = src.get("bootstrap_value")
    gm, lm = prm["gamma"], prm["lambda_"]
    rho_bar, c_bar = prm["rho_bar"], prm["c_bar"]
    if est == "gae":
        return {"out": oracle.gae(src["rewards"], src["values"], src["terminateds"], gm, lm, B, **tr)}
    if est == "lambda_returns":
        return {"out": oracle.lambda_returns(src["rewards"], src["values"], src["terminateds"], gm,
                                             lm, B, **tr)}
    if est == "discounted_returns":
        return {"out": oracle.discounted_returns(src["rewards"], src["terminateds"], gm, B, **tr)}
    if est == "vtrace":
        vs, pg = oracle.vtrace(src["rewards"], src["values"], src["log_rhos"], src["terminateds"],
                               gm, lm, rho_bar, c_bar, B, **tr)
        return {"vs": vs, "pg": pg}
    if est == "retrace":
        return {"out": oracle.retrace(src["rewards"], src["values"], src["q_values"],
                                      src["log_rhos"], src["terminateds"], gm, lm, c_bar,
                                      B, **tr)}
    if est == "eligibility_traces":
        return {"out": oracle.eligibility_traces(src["x"], src["terminateds"], gm, lm)}
    if est == "episodic_prefix_sum":
        return {"out": oracle.episodic_prefix_sum(src["x_int"], src["terminateds"])}
    raise ValueError(est)


def compare(est, got, want, tol, tag=""):
    for key, ref in want.items():
        g = got[key]
        g = g.cpu().numpy() if hasattr(g, "cpu") else np.asarray(g)
        if est == "episodic_prefix_sum":
            bad = np.argwhere(g != ref)
            assert bad.size == 0, "%s%s: %d int32 mismatches, first at %s: %d vs %d" % (
                est, tag, len(bad), tuple(bad[0]), g[tuple(bad[0])], ref[tuple(bad[0])])
            continue
        g = g.astype(np.float64)
        err = np.abs(g - ref) / np.maximum(1.0, np.abs(ref))
        worst = np.unravel_index(np.argmax(err), err.shape) if err.size else None
        assert np.all(np.isfinite(g)), "%s.%s%s: non-finite output" % (est, key, tag)
        assert err.size == 0 or err.max() <= tol, (
            "%s.%s%s: max scaled error %.3g at %s (gpu %.9g, oracle %.9g)"
            % (est, key, tag, err.max(), worst, g[worst], ref[worst]))


def params_of(w):
    return dict(gamma=w.gamma, lambda_=w.lambda_, rho_bar=w.rho_bar, c_bar=w.c_bar)
