"""GPU parity beyond 2^31 elements per array: every offset past the first
2^31 elements needs 64-bit index arithmetic, in each launch shape.

Inputs are drawn in device memory (synthetic_rollouts.device_rollout: 8.6 GB
per float array). Rows are independent, so the oracle checks sampled rows one
by one: the first and last rows and the rows on either side of the 2^31-
element offset. Shapes: the warp rows (T = 128), the register tiles (T =
16388: the last tile of each row is partial, so its later warps' spans lie
wholly past the row end) and the time-major layout ([T, N]: T = 128, and 9
environments over 2^28 steps in 8-environment chunks, checked whole).
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic_rollouts import device_rollout
from tests.parity_common import TOL, compare

pytestmark = pytest.mark.gpu

LIMIT = 1 << 31
GAMMA, LAM = 0.99, 0.95


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    return rl


@pytest.fixture(autouse=True)
def free_memory():
    torch.cuda.empty_cache()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def sample_rows(N, T):
    cross = LIMIT // T
    return sorted({0, 1, N // 3, cross - 1, cross, cross + 1, N - 2, N - 1})


def host(t, rows):
    return t[rows].cpu().numpy()


@pytest.mark.parametrize("N,T", [((1 << 24) + 5, 128), (131075, 16388)])
def test_row_major_past_two_to_the_31(rl, N, T):
    assert N * T > LIMIT
    dev = torch.device("cuda:0")
    g = device_rollout(torch, N, T, 9100 + T, 0.01,
                       ("rewards", "values", "terminateds", "bootstrap_value"), dev)
    rows = sample_rows(N, T)
    r, v, d = (host(g[k], rows) for k in ("rewards", "values", "terminateds"))
    B = g["bootstrap_value"][rows].cpu().numpy()
    out = rl.rlcs_gae(g["rewards"], g["values"], g["terminateds"], GAMMA, LAM,
                      g["bootstrap_value"])
    compare("gae", {"out": host(out, rows)},
            {"out": oracle.gae(r, v, d, GAMMA, LAM, B)}, TOL, " [%dx%d]" % (N, T))
    del out, g["values"]
    out = rl.rlcs_discounted_returns(g["rewards"], g["terminateds"], GAMMA, g["bootstrap_value"])
    compare("discounted_returns", {"out": host(out, rows)},
            {"out": oracle.discounted_returns(r, d, GAMMA, B)}, TOL, " [%dx%d]" % (N, T))
    del out, g["rewards"]
    x = device_rollout(torch, N, T, 9200 + T, 0.0, ("x_int",), dev)["x_int"]
    out = rl.rlcs_episodic_prefix_sum(x, g["terminateds"])
    compare("episodic_prefix_sum", {"out": host(out, rows)},
            {"out": oracle.episodic_prefix_sum(host(x, rows), d)}, TOL)
    del out, x
    x = device_rollout(torch, N, T, 9300 + T, 0.0, ("x",), dev)["x"]
    out = rl.rlcs_eligibility_traces(x, g["terminateds"], GAMMA, LAM)
    compare("eligibility_traces", {"out": host(out, rows)},
            {"out": oracle.eligibility_traces(host(x, rows), d, GAMMA, LAM)}, TOL)
    rl.check_all_workspaces()


def test_time_major_past_two_to_the_31(rl):
    N, T = (1 << 24) + 5, 128
    assert N * T > LIMIT
    dev = torch.device("cuda:0")
    g = device_rollout(torch, N, T, 9400, 0.01,
                       ("rewards", "values", "terminateds", "bootstrap_value"), dev,
                       time_major=True)
    # environments whose last steps lie past the 2^31-element offset
    cross = LIMIT - (T - 1) * N
    envs = sorted({0, 1, N // 2, cross - 1, cross, cross + 1, N - 2, N - 1})
    cols = {k: g[k][:, envs].T.cpu().numpy() for k in ("rewards", "values", "terminateds")}
    B = g["bootstrap_value"][envs].cpu().numpy()
    out = rl.rlcs_gae_tm(g["rewards"], g["values"], g["terminateds"], GAMMA, LAM,
                         g["bootstrap_value"])
    compare("gae", {"out": out[:, envs].T.cpu().numpy()},
            {"out": oracle.gae(cols["rewards"], cols["values"], cols["terminateds"], GAMMA,
                                   LAM, B)}, TOL, " [tm %dx%d]" % (T, N))
    del out
    vs, pg = rl.rlcs_vtrace_tm(g["rewards"], g["values"], g["values"], g["terminateds"], GAMMA,
                               LAM, 1.0, 1.0, g["bootstrap_value"])
    ovs, opg = oracle.vtrace(cols["rewards"], cols["values"], cols["values"],
                                 cols["terminateds"], GAMMA, LAM, 1.0, 1.0, B)
    compare("vtrace", {"vs": vs[:, envs].T.cpu().numpy(), "pg": pg[:, envs].T.cpu().numpy()},
            {"vs": ovs, "pg": opg}, TOL, " [tm %dx%d]" % (T, N))
    rl.check_all_workspaces()


def test_time_major_few_environments_past_two_to_the_31(rl):
    # The 8-environment chunks (N <= 256, T >= 2048) with the four-predecessor
    # look-back window: 9 environments (a full group and a partial one) over
    # 2^28 steps, so every step from t = 2^31 / 9 on lies past the 2^31-element
    # offset. Both environments checked whole, GAE (four arrays, 3 blocks/SM)
    # and discounted returns (three arrays, 4 blocks/SM).
    N, T = 9, 1 << 28
    assert N * T > LIMIT
    dev = torch.device("cuda:0")
    g = device_rollout(torch, N, T, 9500, 0.001,
                       ("rewards", "values", "terminateds", "bootstrap_value"), dev,
                       time_major=True)
    envs = [0, N - 1]
    cols = {k: g[k][:, envs].T.cpu().numpy() for k in ("rewards", "values", "terminateds")}
    B = g["bootstrap_value"][envs].cpu().numpy()
    out = rl.rlcs_gae_tm(g["rewards"], g["values"], g["terminateds"], GAMMA, LAM,
                         g["bootstrap_value"])
    compare("gae", {"out": out[:, envs].T.cpu().numpy()},
            {"out": oracle.gae(cols["rewards"], cols["values"], cols["terminateds"], GAMMA,
                               LAM, B)}, TOL, " [tm %dx%d]" % (T, N))
    del out
    out = rl.rlcs_discounted_returns_tm(g["rewards"], g["terminateds"], GAMMA,
                                        g["bootstrap_value"])
    compare("discounted_returns", {"out": out[:, envs].T.cpu().numpy()},
            {"out": oracle.discounted_returns(cols["rewards"], cols["terminateds"], GAMMA, B)},
            TOL, " [tm %dx%d]" % (T, N))
    del out
    rl.check_all_workspaces()
