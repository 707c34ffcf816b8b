"""GPU parity for rlcs_run_group: several calls in one launch per class.
Every call must meet the float64 oracle at the usual bar; short-row calls
must also agree with their namesake's lone call to 1e-6 relative (the same
body runs, compiled into another kernel), and every prefix sum bit for bit. Covers all eight groupable estimators in one
group, mixed row lengths (all three strip classes and long rows, some
chained by look-back) with and without truncation in one call list, ragged
N, V-trace without pg, a full group of 16 calls, repeat calls on one
workspace, the cross-call overlap check, and capture in a CUDA graph."""
import numpy as np
import pytest
import torch

from synthetic_rollouts import rollout
from tests.parity_common import TOL, compare, run_oracle, to_dev

pytestmark = pytest.mark.gpu

PRM = dict(gamma=0.99, lambda_=0.95, rho_bar=1.0, c_bar=1.0)


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    return rl


def group_args(est, g, trunc, prm=PRM):
    tr = dict(truncateds=g["truncateds"], next_values=g["next_values"]) if trunc else {}
    gm, lm = prm["gamma"], prm["lambda_"]
    B = g["bootstrap_value"]
    if est in ("gae", "lambda_returns", "gae_and_returns"):
        return dict(rewards=g["rewards"], values=g["values"], terminateds=g["terminateds"],
                    gamma=gm, lambda_=lm, bootstrap_value=B, **tr)
    if est == "discounted_returns":
        return dict(rewards=g["rewards"], terminateds=g["terminateds"], gamma=gm,
                    bootstrap_value=B, **tr)
    if est == "vtrace":
        return dict(rewards=g["rewards"], values=g["values"], log_rhos=g["log_rhos"],
                    terminateds=g["terminateds"], gamma=gm, lambda_=lm,
                    rho_bar=prm["rho_bar"], c_bar=prm["c_bar"], bootstrap_value=B, **tr)
    if est == "retrace":
        return dict(rewards=g["rewards"], values=g["values"], q_values=g["q_values"],
                    log_rhos=g["log_rhos"], terminateds=g["terminateds"], gamma=gm, lambda_=lm,
                    c_bar=prm["c_bar"], bootstrap_value=B, **tr)
    if est == "eligibility_traces":
        return dict(x=g["x"], dones=g["terminateds"], gamma=gm, lambda_=lm)
    if est == "episodic_prefix_sum":
        return dict(x=g["x_int"], dones=g["terminateds"])
    raise ValueError(est)


def alone(rl, est, kw):
    f = getattr(rl, "rlcs_" + est)
    kw = dict(kw)
    if est in ("eligibility_traces", "episodic_prefix_sum"):
        return f(kw.pop("x"), kw.pop("dones"), **kw)
    return f(**kw)


def as_dict(est, res):
    if est == "vtrace":
        return {"vs": res[0], "pg": res[1]}
    if est == "gae_and_returns":
        return {"adv": res[0], "ret": res[1]}
    return {"out": res}


def oracle_of(est, src, trunc):
    if est == "gae_and_returns":
        return {"adv": run_oracle("gae", src, PRM, trunc)["out"],
                "ret": run_oracle("lambda_returns", src, PRM, trunc)["out"]}
    return run_oracle(est, src, PRM, trunc)


ALL = ("gae", "lambda_returns", "discounted_returns", "vtrace", "retrace", "eligibility_traces",
       "episodic_prefix_sum", "gae_and_returns")


def check(rl, plan):
    """plan: list of (est, N, T, trunc, seed). Runs them as one group and alone."""
    dev = torch.device("cuda:0")
    calls, srcs = [], []
    for est, N, T, trunc, seed in plan:
        src = rollout(N, T, seed, p_term=0.02, p_trunc=0.01 if trunc else 0.0)
        g = to_dev(src, dev)
        calls.append((est, group_args(est, g, trunc)))
        srcs.append(src)
    got = rl.rlcs_run_group(calls)
    torch.cuda.synchronize()
    for (est, N, T, trunc, seed), (_, kw), res, src in zip(plan, calls, got, srcs):
        tag = " [%s N=%d T=%d trunc=%s]" % (est, N, T, trunc)
        mine = as_dict(est, res)
        # Short rows: the group runs the warp-row body of the lone call,
        # compiled into another kernel, so the lone call is forced to that
        # shape (by itself a light call may take the eight-step tiles, whose
        # combination order differs). The integer prefix sum repeats bit for
        # bit; floats may round differently where the compiler fuses
        # multiply-adds differently, so they must agree to a few ulps. Long
        # rows are chained by look-back, whose combination order varies:
        # they are held to the oracle only.
        if T <= 512:
            rl.rlcs_set_shape_override(rl.RLCS_SHAPE_WARP_ROW, 0)
        try:
            ref = as_dict(est, alone(rl, est, kw))
        finally:
            rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
        for k in mine:
            if est == "episodic_prefix_sum":
                assert torch.equal(mine[k], ref[k]), "group differs from the lone call" + tag
            elif T <= 512:
                diff = (mine[k] - ref[k]).abs() / ref[k].abs().clamp(min=1.0)
                assert float(diff.max()) <= 1e-6, "group differs from the lone call" + tag
        compare("episodic_prefix_sum" if est == "episodic_prefix_sum" else est, mine,
                oracle_of(est, src, trunc), TOL, tag)


def test_all_estimators_one_group(rl):
    check(rl, [(e, 4096, 128, False, 100 + i) for i, e in enumerate(ALL)])


def test_mixed_classes_and_ragged_sizes(rl):
    plan = []
    sizes = [(7, 1), (33, 100), (1000, 129), (5, 256), (64, 300), (3, 512), (129, 77)]
    for i, est in enumerate(ALL):
        N, T = sizes[i % len(sizes)]
        plan.append((est, N, T, i % 2 == 1 and est not in ("eligibility_traces",
                                                            "episodic_prefix_sum"), 200 + i))
    check(rl, plan)
    check(rl, [(e, 333, 512, True, 300 + i) for i, e in enumerate(ALL[:5])])


def test_full_group_of_sixteen(rl):
    check(rl, [(ALL[i % len(ALL)], 100 + 17 * i, 64 + 29 * i, i % 3 == 0 and
                ALL[i % len(ALL)] not in ("eligibility_traces", "episodic_prefix_sum"), 400 + i)
               for i in range(16)])


def test_vtrace_without_pg(rl):
    src = rollout(64, 128, 500, p_term=0.02)
    g = to_dev(src, torch.device("cuda:0"))
    kw = dict(group_args("vtrace", g, False), with_pg=False)
    (vs, pg), = rl.rlcs_run_group([("vtrace", kw)])
    assert pg is None
    compare("vtrace", {"vs": vs}, {"vs": run_oracle("vtrace", src, PRM, False)["vs"]}, TOL)


def test_overlapping_calls_are_rejected(rl):
    src = rollout(64, 128, 501, p_term=0.02)
    g = to_dev(src, torch.device("cuda:0"))
    a = group_args("gae", g, False)
    b = dict(group_args("discounted_returns", g, False), out=g["rewards"])  # writes a's input
    with pytest.raises(rl.RlcsError):
        rl.rlcs_run_group([("gae", a), ("discounted_returns", b)])


def test_group_in_cuda_graph(rl):
    dev = torch.device("cuda:0")
    src = rollout(512, 128, 502, p_term=0.02)
    g = to_dev(src, dev)
    outs = {e: (torch.empty(512, 128, device=dev, dtype=torch.int32)
                if e == "episodic_prefix_sum" else torch.empty(512, 128, device=dev))
            for e in ALL}
    extra = {"vtrace": torch.empty(512, 128, device=dev),
             "gae_and_returns": torch.empty(512, 128, device=dev)}
    calls = []
    for e in ALL:
        kw = dict(group_args(e, g, False), out=outs[e])
        if e == "vtrace":
            kw["out_pg"] = extra[e]
        if e == "gae_and_returns":
            kw["out_returns"] = extra[e]
        calls.append((e, kw))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rl.rlcs_run_group(calls, stream=s)  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rl.rlcs_run_group(calls, stream=s)
    for o in list(outs.values()) + list(extra.values()):
        o.zero_()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    for e in ALL:
        res = outs[e]
        if e == "vtrace":
            res = (outs[e], extra[e])
        if e == "gae_and_returns":
            res = (outs[e], extra[e])
        compare(e if e != "gae_and_returns" else "gae_and_returns", as_dict(e, res),
                oracle_of(e, src, False), TOL)


def test_long_rows_one_group(rl):
    # one tile per row (4096 steps) and chained tiles (20000 steps)
    check(rl, [(e, 256, 4096, False, 600 + i) for i, e in enumerate(ALL)])
    check(rl, [(e, 48, 20000, e not in ("eligibility_traces", "episodic_prefix_sum"), 700 + i)
               for i, e in enumerate(ALL)])


def test_short_and_long_rows_mixed(rl):
    sizes = [(4096, 128), (7, 5000), (300, 513), (33, 1024), (129, 16384), (5, 1025),
             (1000, 77), (64, 9000)]
    check(rl, [(e, N, T, i % 2 == 0 and e not in ("eligibility_traces", "episodic_prefix_sum"),
                800 + i) for i, (e, (N, T)) in enumerate(zip(ALL, sizes))])


def test_long_group_repeats_on_one_workspace(rl):
    # the shared workspace moves to a new epoch after every launch
    plan = [(e, 32, 12000, False, 900 + i) for i, e in enumerate(ALL)]
    for _ in range(3):
        check(rl, plan)
    rl.check_all_workspaces()


def test_more_than_sixteen_calls_run_as_consecutive_groups(rl):
    check(rl, [(ALL[i % len(ALL)], 20 + i, 100 + 13 * i, False, 1000 + i) for i in range(21)])


def test_long_row_group_in_cuda_graph(rl):
    dev = torch.device("cuda:0")
    src = rollout(40, 9000, 1100, p_term=0.002)
    g = to_dev(src, dev)
    ests = ("gae", "vtrace", "episodic_prefix_sum")
    outs, calls = {}, []
    for e in ests:
        kw = group_args(e, g, False)
        outs[e] = torch.empty(40, 9000, device=dev,
                              dtype=torch.int32 if e == "episodic_prefix_sum" else torch.float32)
        kw["out"] = outs[e]
        if e == "vtrace":
            outs["pg"] = torch.empty(40, 9000, device=dev)
            kw["out_pg"] = outs["pg"]
        calls.append((e, kw))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rl.rlcs_run_group(calls, stream=s)  # warm-up: workspace allocated outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rl.rlcs_run_group(calls, stream=s)
    for _ in range(3):
        for o in outs.values():
            o.zero_()
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        compare("gae", {"out": outs["gae"]}, oracle_of("gae", src, False), TOL)
        compare("vtrace", {"vs": outs["vtrace"], "pg": outs["pg"]},
                oracle_of("vtrace", src, False), TOL)
        compare("episodic_prefix_sum", {"out": outs["episodic_prefix_sum"]},
                oracle_of("episodic_prefix_sum", src, False), TOL)
    rl.check_all_workspaces()
