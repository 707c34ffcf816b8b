"""Parity in the launch configuration the benchmark times.

bench.py's headline step runs the seven estimators at 4096 x 128 on seven
streams (fork/join) inside CUDA graphs of whole steps, each step on its own
rotating buffer set. This test builds the step with bench.py's own helpers
(buffer sets, launch and group arguments), captures and replays it, and
compares every output of every buffer set with the float64 oracle; it does
the same for the grouped schedule (one rlcs_run_group call per step) and
for the truncated five. Same bar as the other parity tests.
"""
import os
import sys

import pytest
import torch

from synthetic_rollouts import WORKLOADS, rollout
from tests.parity_common import TOL, compare, params_of, run_oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NSETS, STEPS = 3, 5


@pytest.fixture(scope="module")
def env():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    import linear_recurrence_scan_affine_gb300 as rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    return bench, rl, torch.device("cuda:0")


def _outputs(bench, est, e):
    return {o: e[o] for o in bench.SPECS[est][1]}


def _check(bench, rl, sets, src, prm, ests, trunc):
    for i, st in enumerate(sets):
        for est in ests:
            base = bench.base_name(est)
            want = run_oracle(base, src, prm, trunc)
            got = _outputs(bench, est, st[est])
            compare(base, got, want, TOL, " [bench set %d, %s]" % (i, est))
    rl.check_all_workspaces()


def _rollout(name):
    w = WORKLOADS[name]
    return w, rollout(w.N, w.T, w.seed, w.p_term, w.p_trunc), params_of(w)


def test_seven_streams_graph_as_in_the_bench(env):
    bench, rl, dev = env
    w, src, prm = _rollout("all7_4096x128")
    order = list(bench.ESTIMATORS)
    sets = bench.make_sets(torch, rl, src, dev, NSETS, order)
    for st in sets:  # poison the outputs: every one must be written
        for est in order:
            for o in bench.SPECS[est][1]:
                out = st[est][o]
                out.fill_(float("nan") if out.dtype == torch.float32 else -1)
    stream = torch.cuda.Stream(dev)
    side = {est: torch.cuda.Stream(dev) for est in order}
    for s_ in [stream] + list(side.values()):  # set-up call on every stream, outside capture
        s_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_):
            for est in order:
                bench.launch(rl, est, sets[0][est], prm)
    torch.cuda.synchronize()

    def steps():
        for est in order:
            side[est].wait_stream(stream)
            with torch.cuda.stream(side[est]):
                for i in range(STEPS):
                    bench.launch(rl, est, sets[i % NSETS][est], prm)
        for est in order:
            stream.wait_stream(side[est])

    g = bench.capture(torch, stream, steps)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    _check(bench, rl, sets, src, prm, order, False)


def test_grouped_step_as_in_the_bench(env):
    bench, rl, dev = env
    w, src, prm = _rollout("all7_4096x128")
    order = list(bench.ESTIMATORS)
    sets = bench.make_sets(torch, rl, src, dev, NSETS, order)
    stream = torch.cuda.Stream(dev)
    calls = [[(est, bench.group_kwargs(est, st[est], prm)) for est in order] for st in sets]
    with torch.cuda.stream(stream):
        rl.rlcs_run_group(calls[0])
    torch.cuda.synchronize()
    g = bench.capture(torch, stream, lambda: [rl.rlcs_run_group(calls[i % NSETS])
                                              for i in range(STEPS)])
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    _check(bench, rl, sets, src, prm, order, False)


def test_truncated_five_on_streams_as_in_the_bench(env):
    bench, rl, dev = env
    w, src, prm = _rollout("trunc5_4096x128")
    ests = [e + "_trunc" for e in w.estimators]
    sets = bench.make_sets(torch, rl, src, dev, NSETS, ests)
    stream = torch.cuda.Stream(dev)
    side = {est: torch.cuda.Stream(dev) for est in ests}
    for s_ in [stream] + list(side.values()):
        s_.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s_):
            for est in ests:
                bench.launch(rl, est, sets[0][est], prm)
    torch.cuda.synchronize()

    def steps():
        for est in ests:
            side[est].wait_stream(stream)
            with torch.cuda.stream(side[est]):
                for i in range(STEPS):
                    bench.launch(rl, est, sets[i % NSETS][est], prm)
        for est in ests:
            stream.wait_stream(side[est])

    g = bench.capture(torch, stream, steps)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    _check(bench, rl, sets, src, prm, ests, True)
