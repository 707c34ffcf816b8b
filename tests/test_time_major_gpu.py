"""GPU parity for the time-major [T, N] entry points (the _tm functions).

Inputs are drawn [N, T] as everywhere else, transposed to [T, N] for the
GPU, and the outputs transposed back and compared element by element with
the float64 oracle at the usual bar (1e-4 relative; the prefix sum
bit-exact). A block owns 32 environments and one chunk of T (128 steps),
or, with at most 256 environments and T >= 2048, 8 environments and 512 or
1024 steps; chunks of the same environments are linked by a look-back through
the workspace, which reads one predecessor per warp and round or, for few
8-environment groups with long chains, four. Sizes cover ragged environment
groups (N not a multiple of 32 or 8), exact group and chunk edges, ragged
and many-chunk T (chains of up to 1024 chunks), both warp shapes (8-step
spans below T = 1024, 16-step spans from there), both block shapes, both
look-back windows (13 x 20000 and 100 x 40000 take four distances per warp,
with a partial last group), truncations and the degenerate T = 1.
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic_rollouts import affine_inputs, rollout
from tests.parity_common import TOL, TOL_VLONG, compare

pytestmark = pytest.mark.gpu

SIZES = [(4096, 128), (1000, 300), (7, 1), (33, 129), (256, 1030), (9, 4097), (32, 128),
         (31, 129), (64, 16384), (48, 1023), (5, 2048), (100, 2600), (255, 9001), (257, 2048),
         (200, 20000), (17, 3000), (13, 20000), (100, 40000)]
PRM = dict(gamma=0.99, lambda_=0.95, rho_bar=1.0, c_bar=1.0)


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    return rl


def tm(a, dev=torch.device("cuda:0")):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a).T)).to(dev)


def back(t):
    return t.cpu().numpy().T


@pytest.mark.parametrize("N,T", SIZES)
@pytest.mark.parametrize("trunc", [False, True])
def test_backward_estimators_time_major(rl, N, T, trunc):
    src = rollout(N, T, 11000 + N + T, p_term=0.01, p_trunc=0.005 if trunc else 0.0)
    g = {k: (tm(v) if v.ndim == 2 else torch.from_numpy(v).cuda()) for k, v in src.items()}
    kw = dict(truncateds=g["truncateds"], next_values=g["next_values"]) if trunc else {}
    kwn = dict(truncateds=src["truncateds"], next_values=src["next_values"]) if trunc else {}
    B, Bn = g["bootstrap_value"], src["bootstrap_value"]
    r, v, d = g["rewards"], g["values"], g["terminateds"]
    rn, vn, dn = src["rewards"], src["values"], src["terminateds"]
    gm, lm = PRM["gamma"], PRM["lambda_"]
    compare("gae", {"out": back(rl.rlcs_gae_tm(r, v, d, gm, lm, B, **kw))},
            {"out": oracle.gae(rn, vn, dn, gm, lm, Bn, **kwn)}, TOL)
    compare("lambda_returns", {"out": back(rl.rlcs_lambda_returns_tm(r, v, d, gm, lm, B, **kw))},
            {"out": oracle.lambda_returns(rn, vn, dn, gm, lm, Bn, **kwn)}, TOL)
    compare("discounted_returns",
            {"out": back(rl.rlcs_discounted_returns_tm(r, d, gm, B, **kw))},
            {"out": oracle.discounted_returns(rn, dn, gm, Bn, **kwn)}, TOL)
    vs, pg = rl.rlcs_vtrace_tm(r, v, g["log_rhos"], d, gm, lm, 1.0, 1.0, B, **kw)
    ovs, opg = oracle.vtrace(rn, vn, src["log_rhos"], dn, gm, lm, 1.0, 1.0, Bn, **kwn)
    compare("vtrace", {"vs": back(vs), "pg": back(pg)}, {"vs": ovs, "pg": opg}, TOL)
    compare("retrace",
            {"out": back(rl.rlcs_retrace_tm(r, v, g["q_values"], g["log_rhos"], d, gm, lm, 1.0,
                                            B, **kw))},
            {"out": oracle.retrace(rn, vn, src["q_values"], src["log_rhos"], dn, gm, lm, 1.0,
                                   Bn, **kwn)}, TOL)
    adv, ret = rl.rlcs_gae_and_returns_tm(r, v, d, gm, lm, B, **kw)
    compare("gae", {"out": back(adv)}, {"out": oracle.gae(rn, vn, dn, gm, lm, Bn, **kwn)}, TOL)
    compare("lambda_returns", {"out": back(ret)},
            {"out": oracle.lambda_returns(rn, vn, dn, gm, lm, Bn, **kwn)}, TOL)


@pytest.mark.parametrize("N,T", SIZES)
def test_forward_estimators_time_major(rl, N, T):
    src = rollout(N, T, 12000 + N + T, p_term=0.02)
    d = tm(src["terminateds"])
    got = back(rl.rlcs_eligibility_traces_tm(tm(src["x"]), d, 0.9, 0.8))
    compare("eligibility_traces", {"out": got},
            {"out": oracle.eligibility_traces(src["x"], src["terminateds"], 0.9, 0.8)}, TOL)
    got = back(rl.rlcs_episodic_prefix_sum_tm(tm(src["x_int"]), d))
    assert np.array_equal(got, oracle.episodic_prefix_sum(src["x_int"], src["terminateds"]))


@pytest.mark.parametrize("N,T", SIZES)
@pytest.mark.parametrize("reverse", [False, True])
def test_affine_scan_time_major(rl, N, T, reverse):
    src = affine_inputs(N, T, 13000 + N + T)
    got = back(rl.rlcs_affine_scan_tm(tm(src["a"]), tm(src["b"]), tm(src["reset"]),
                                      torch.from_numpy(src["x_init"]).cuda(), reverse=reverse))
    want = oracle.affine_scan(src["a"], src["b"], src["reset"], src["x_init"], reverse=reverse)
    compare("affine_scan", {"out": got}, {"out": want}, TOL)


def test_very_long_time_major_rows(rl):
    # 1024 chunks per environment: the longest look-back chains
    N, T = 8, 131072
    src = rollout(N, T, 14000, p_term=1e-4)
    g = {k: (tm(v) if v.ndim == 2 else torch.from_numpy(v).cuda()) for k, v in src.items()}
    got = back(rl.rlcs_gae_tm(g["rewards"], g["values"], g["terminateds"], 0.999, 1.0,
                              g["bootstrap_value"]))
    want = oracle.gae(src["rewards"], src["values"], src["terminateds"], 0.999, 1.0,
                      src["bootstrap_value"])
    compare("gae", {"out": got}, {"out": want}, TOL_VLONG)
    vs, pg = rl.rlcs_vtrace_tm(g["rewards"], g["values"], g["log_rhos"], g["terminateds"],
                               0.999, 1.0, 1.0, 1.0, g["bootstrap_value"])
    ovs, opg = oracle.vtrace(src["rewards"], src["values"], src["log_rhos"], src["terminateds"],
                             0.999, 1.0, 1.0, 1.0, src["bootstrap_value"])
    compare("vtrace", {"vs": back(vs), "pg": back(pg)}, {"vs": ovs, "pg": opg}, TOL_VLONG)


def test_time_major_repeat_calls(rl):
    # The workspace moves to a new epoch after every chained launch. Every
    # repeat must meet the oracle; the last bits of float results may differ
    # with the point where a look-back found an inclusive value, so only the
    # integer path is required to repeat bit for bit.
    N, T = 1000, 3000
    src = rollout(N, T, 15000, p_term=0.01, p_trunc=0.005)
    g = {k: (tm(v) if v.ndim == 2 else torch.from_numpy(v).cuda()) for k, v in src.items()}
    kw = dict(truncateds=g["truncateds"], next_values=g["next_values"])
    want = oracle.retrace(src["rewards"], src["values"], src["q_values"], src["log_rhos"],
                          src["terminateds"], 0.99, 0.95, 1.0, src["bootstrap_value"],
                          truncateds=src["truncateds"], next_values=src["next_values"])
    for _ in range(3):
        got = rl.rlcs_retrace_tm(g["rewards"], g["values"], g["q_values"], g["log_rhos"],
                                 g["terminateds"], 0.99, 0.95, 1.0, g["bootstrap_value"], **kw)
        compare("retrace", {"out": back(got)}, {"out": want}, TOL)
    first = rl.rlcs_episodic_prefix_sum_tm(g["x_int"], g["terminateds"]).clone()
    for _ in range(3):
        assert torch.equal(rl.rlcs_episodic_prefix_sum_tm(g["x_int"], g["terminateds"]), first)
    rl.check_all_workspaces()


def test_time_major_cuda_graph_capture_and_replay(rl):
    # chained chunks inside a captured graph: every replay moves the
    # workspace to a new epoch
    N, T = 200, 3000
    src = rollout(N, T, 16000, p_term=0.01, p_trunc=0.005)
    g = {k: (tm(v) if v.ndim == 2 else torch.from_numpy(v).cuda()) for k, v in src.items()}
    kw = dict(truncateds=g["truncateds"], next_values=g["next_values"])
    out = torch.empty_like(g["rewards"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up: the stream's workspace exists before capture
        rl.rlcs_gae_tm(g["rewards"], g["values"], g["terminateds"], 0.99, 0.95,
                       g["bootstrap_value"], out=out, stream=s, **kw)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rl.rlcs_gae_tm(g["rewards"], g["values"], g["terminateds"], 0.99, 0.95,
                       g["bootstrap_value"], out=out, stream=s, **kw)
    want = oracle.gae(src["rewards"], src["values"], src["terminateds"], 0.99, 0.95,
                      src["bootstrap_value"], truncateds=src["truncateds"],
                      next_values=src["next_values"])
    for _ in range(4):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        compare("gae", {"out": back(out)}, {"out": want}, TOL)
    rl.check_all_workspaces()


@pytest.mark.parametrize("name", ["longT_256x4096", "longT_256x16384"])
def test_time_major_long_row_recipes(rl, name):
    # the long-row recipes with their own scalars (gamma = 0.997, lambda = 0.95),
    # stored time-major
    from synthetic_rollouts import WORKLOADS, workload_inputs
    w = WORKLOADS[name]
    src = workload_inputs(w)
    g = {k: (tm(v) if v.ndim == 2 else torch.from_numpy(v).cuda()) for k, v in src.items()}
    gm, lm, B, Bn = w.gamma, w.lambda_, g["bootstrap_value"], src["bootstrap_value"]
    r, v, d = g["rewards"], g["values"], g["terminateds"]
    rn, vn, dn = src["rewards"], src["values"], src["terminateds"]
    compare("discounted_returns", {"out": back(rl.rlcs_discounted_returns_tm(r, d, gm, B))},
            {"out": oracle.discounted_returns(rn, dn, gm, Bn)}, TOL)
    compare("gae", {"out": back(rl.rlcs_gae_tm(r, v, d, gm, lm, B))},
            {"out": oracle.gae(rn, vn, dn, gm, lm, Bn)}, TOL)
    compare("lambda_returns", {"out": back(rl.rlcs_lambda_returns_tm(r, v, d, gm, lm, B))},
            {"out": oracle.lambda_returns(rn, vn, dn, gm, lm, Bn)}, TOL)
    vs, pg = rl.rlcs_vtrace_tm(r, v, g["log_rhos"], d, gm, lm, 1.0, 1.0, B)
    ovs, opg = oracle.vtrace(rn, vn, src["log_rhos"], dn, gm, lm, 1.0, 1.0, Bn)
    compare("vtrace", {"vs": back(vs), "pg": back(pg)}, {"vs": ovs, "pg": opg}, TOL)
    compare("eligibility_traces",
            {"out": back(rl.rlcs_eligibility_traces_tm(tm(src["x"]), d, gm, lm))},
            {"out": oracle.eligibility_traces(src["x"], dn, gm, lm)}, TOL)
    rl.check_all_workspaces()


@pytest.mark.parametrize("N,T", [(4096, 128), (64, 16384), (256, 16384), (1024, 4096)])
@pytest.mark.parametrize("shift", [1, 2])
def test_time_major_inputs_off_16_byte_boundaries(rl, N, T, shift):
    # Every time-major shape prefetches its chunk's rows into L2 in 16-byte
    # aligned pieces and skips an input whose base is off that boundary; the
    # loads themselves take any 4-byte aligned array. Inputs start 4 or 8
    # bytes into their allocation (the short, 8- and 32-environment shapes;
    # GAE moves four arrays, discounted returns three).
    src = rollout(N, T, 14000 + N + T + shift, p_term=0.01)

    def shifted(a):
        flat = torch.empty(N * T + shift, dtype=torch.float32, device="cuda")
        view = flat[shift:].view(T, N)
        view.copy_(tm(a))
        assert view.data_ptr() % 16 == 4 * shift % 16
        return view

    r, v, d = shifted(src["rewards"]), shifted(src["values"]), shifted(src["terminateds"])
    B = torch.from_numpy(src["bootstrap_value"]).cuda()
    gm, lm = PRM["gamma"], PRM["lambda_"]
    rn, vn, dn, Bn = src["rewards"], src["values"], src["terminateds"], src["bootstrap_value"]
    compare("gae", {"out": back(rl.rlcs_gae_tm(r, v, d, gm, lm, B))},
            {"out": oracle.gae(rn, vn, dn, gm, lm, Bn)}, TOL)
    compare("discounted_returns", {"out": back(rl.rlcs_discounted_returns_tm(r, d, gm, B))},
            {"out": oracle.discounted_returns(rn, dn, gm, Bn)}, TOL)
