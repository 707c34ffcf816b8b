"""GPU parity: every estimator through the C ABI against the float64 oracle.

Bar: |gpu - oracle| <= 1e-4 * max(1, |oracle|) for T <= 16384 and 1e-3 at
T = 131072; the int32 episodic prefix sum is bit-exact. Covered: every
workload recipe at its full size (with and without truncations), both launch
shapes forced on small ragged sizes that span several strips/chunks and a
ragged tail, unaligned rows (scalar path), degenerate masks, workspace reuse
across calls, and CUDA-graph capture.
"""
import numpy as np
import pytest
import torch

from synthetic_rollouts import WORKLOADS, rollout, workload_inputs
from tests.parity_common import (ALL, BACKWARD, TOL, TOL_VLONG, compare, params_of, run_gpu,
                                 run_oracle, to_dev)

pytestmark = pytest.mark.gpu

DEFAULT = dict(gamma=0.99, lambda_=0.95, rho_bar=1.0, c_bar=1.0)


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    yield rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.fixture
def dev():
    return torch.device("cuda:0")


def check_all(rl, src, g, prm, ests, trunc, tol=TOL, tag=""):
    for est in ests:
        got = run_gpu(rl, est, g, prm, trunc and est in BACKWARD)
        want = run_oracle(est, src, prm, trunc and est in BACKWARD)
        compare(est, got, want, tol, tag)
    rl.check_all_workspaces()


# --------------------------------------------------------------------------
# Every workload recipe at full size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workload_full_size(rl, dev, name):
    w = WORKLOADS[name]
    src = workload_inputs(w)
    g = to_dev(src, dev)
    tol = TOL_VLONG if w.T > 16384 else TOL
    check_all(rl, src, g, params_of(w), w.estimators, w.p_trunc > 0, tol, " [%s]" % name)


@pytest.mark.parametrize("name", ["all7_4096x128", "longT_256x4096", "longT_256x16384",
                                  "vlong_8x131072"])
def test_workload_with_truncations(rl, dev, name):
    w = WORKLOADS[name]
    src = rollout(w.N, w.T, w.seed + 50, w.p_term, p_trunc=max(w.p_term / 2, 0.0005))
    g = to_dev(src, dev)
    ests = [e for e in w.estimators if e in BACKWARD]
    tol = TOL_VLONG if w.T > 16384 else TOL
    check_all(rl, src, g, params_of(w), ests, True, tol, " [%s+trunc]" % name)


# --------------------------------------------------------------------------
# Launch shapes forced on small, ragged sizes
# --------------------------------------------------------------------------

ROW_TS = [1, 2, 3, 4, 5, 64, 127, 128, 129, 200, 255, 256, 257, 300, 511, 512]
CHUNK_CASES = [(1024, T) for T in (1, 7, 1000, 1024, 1028, 3000, 5003)] + \
              [(2048, T) for T in (1024, 2048, 2052, 4100, 9001)] + \
              [(4096, T) for T in (4096, 8192, 12289, 40000)]


@pytest.mark.parametrize("T", ROW_TS)
@pytest.mark.parametrize("trunc", [False, True])
def test_warp_row_shape(rl, dev, T, trunc):
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_WARP_ROW, 0)
    try:
        src = rollout(9, T, 2000 + T, p_term=0.05, p_trunc=0.03 if trunc else 0.0)
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, trunc, tag=" [row T=%d]" % T)
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.mark.parametrize("chunk,T", CHUNK_CASES)
@pytest.mark.parametrize("trunc", [False, True])
@pytest.mark.parametrize("shape", ["chunk", "tile"])
def test_block_shapes(rl, dev, shape, chunk, T, trunc):
    code = rl.RLCS_SHAPE_BLOCK_CHUNK if shape == "chunk" else rl.RLCS_SHAPE_BLOCK_TILE
    rl.rlcs_set_shape_override(code, chunk)
    try:
        src = rollout(5, T, 3000 + T + chunk, p_term=0.01, p_trunc=0.005 if trunc else 0.0)
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, trunc,
                  tag=" [%s=%d T=%d]" % (shape, chunk, T))
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.mark.parametrize("shape", ["chunk", "tile"])
def test_block_shapes_many_rows(rl, dev, shape):
    """Many rows of several tiles each: with row-interleaved tile order a
    tile's predecessor is N blocks back."""
    code = rl.RLCS_SHAPE_BLOCK_CHUNK if shape == "chunk" else rl.RLCS_SHAPE_BLOCK_TILE
    rl.rlcs_set_shape_override(code, 1024)
    try:
        src = rollout(700, 5000, 3100, p_term=0.002, p_trunc=0.001)
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, True, tag=" [%s many rows]" % shape)
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.mark.parametrize("N,T", [(200, 4000), (700, 3001), (40, 9000), (500, 8200)])
def test_sixteen_warp_tiles_one_and_several_waves(rl, dev, N, T):
    """4096-step tiles run as 16 warps of 2 strips, with a second, lighter
    instance for three-array calls whose grid spans more than one wave.
    These sizes (automatic choice for the first two, 4096-step tiles forced
    for the others) take both instances, whole-row tiles (T <= 4096, no
    look-back) and chained ones, with ragged tails."""
    forced = T > 4096
    if forced:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_BLOCK_TILE, 4096)
    try:
        src = rollout(N, T, 3200 + N + T, p_term=0.003, p_trunc=0.002)
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, True, tag=" [16 warps %dx%d]" % (N, T))
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, False, tag=" [16 warps %dx%d]" % (N, T))
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.mark.parametrize("N,T,forced", [(5, 8192, True), (3, 20000, True), (2, 40001, True),
                                        (40, 9000, False), (76, 16384, False)])
def test_thirty_two_warp_tiles(rl, dev, N, T, forced):
    """8192-step tiles (32 warps of 2 strips): forced on ragged rows, and
    taken by the planner where N * ceil(T / 8192) fits in one block per SM."""
    if forced:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_BLOCK_TILE, 8192)
    try:
        src = rollout(N, T, 3400 + N + T, p_term=0.002, p_trunc=0.001)
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, True, tag=" [32 warps %dx%d]" % (N, T))
        check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, False, tag=" [32 warps %dx%d]" % (N, T))
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


@pytest.mark.parametrize("N,T", [(1, 8), (300, 8), (37, 16), (33, 120), (7, 200), (300, 1000),
                                 (5, 2040), (19, 2048), (3, 2056), (3, 3000), (400, 4096),
                                 (41, 6000), (9, 8200), (2, 20000), (300, 6000), (20000, 128),
                                 (37, 132), (3, 1024), (700, 512), (13000, 256), (76, 16384)])
def test_eight_step_tiles_for_light_calls(rl, dev, N, T):
    """Discounted returns takes tiles of eight steps per lane when T % 8 == 0
    (whole rows packed into 2048- or 4096-step tiles, chained tiles beyond,
    both register budgets); rows with T % 8 != 0, unaligned arrays and
    truncated calls take the other shapes. Traces and the prefix sum run
    beside it on the same data (the four-step shapes)."""
    light = ["discounted_returns", "eligibility_traces", "episodic_prefix_sum"]
    src = rollout(N, T, 3300 + N + T, p_term=0.003, p_trunc=0.002)
    check_all(rl, src, to_dev(src, dev), DEFAULT, light, False, tag=" [8-step %dx%d]" % (N, T))
    check_all(rl, src, to_dev(src, dev, offset=1), DEFAULT, light, False,
              tag=" [unaligned %dx%d]" % (N, T))
    check_all(rl, src, to_dev(src, dev), DEFAULT, ["discounted_returns"], True,
              tag=" [truncated %dx%d]" % (N, T))


@pytest.mark.parametrize("shape,chunk,T", [(1, 0, 128), (1, 0, 300), (2, 1024, 3000),
                                           (2, 4096, 9000), (2, 2048, 2048), (3, 1024, 3000),
                                           (3, 4096, 9000), (3, 2048, 2048)])
def test_unaligned_rows_take_scalar_path(rl, dev, shape, chunk, T):
    rl.rlcs_set_shape_override(shape, chunk)
    try:
        src = rollout(6, T, 4000 + T, p_term=0.02, p_trunc=0.01)
        g = to_dev(src, dev, offset=1)
        assert g["rewards"].data_ptr() % 16 != 0
        check_all(rl, src, g, DEFAULT, ALL, True, tag=" [unaligned T=%d]" % T)
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


# --------------------------------------------------------------------------
# Degenerate masks and window edges
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 128, 2500, 20000])
@pytest.mark.parametrize("pattern", ["all_done", "no_done", "done_first", "done_last",
                                     "trunc_everywhere"])
def test_degenerate_masks(rl, dev, T, pattern):
    src = rollout(3, T, 5000 + T, p_term=0.0, p_trunc=0.01)
    d, tr = src["terminateds"], src["truncateds"]
    tr[:] = 0
    if pattern == "all_done":
        d[:] = 1
    elif pattern == "done_first":
        d[:, 0] = 1
    elif pattern == "done_last":
        d[:, -1] = 1
    elif pattern == "trunc_everywhere":
        tr[:] = 1
    check_all(rl, src, to_dev(src, dev), DEFAULT, ALL, True, tag=" [%s T=%d]" % (pattern, T))


def test_both_masks_set_termination_wins(rl, dev):
    src = rollout(4, 700, 77, p_term=0.05, p_trunc=0.0)
    src["truncateds"] = src["terminateds"].copy()        # every terminated step also truncated
    src["truncateds"][:, ::37] = 1.0
    src["next_values"] = rollout(4, 700, 78, 0.0)["values"]
    check_all(rl, src, to_dev(src, dev), DEFAULT, BACKWARD, True, tag=" [both masks]")


def test_no_bootstrap_and_no_pg(rl, dev):
    src = rollout(7, 1500, 79, p_term=0.01)
    g = to_dev(src, dev)
    src.pop("bootstrap_value")
    g.pop("bootstrap_value")
    check_all(rl, src, g, DEFAULT, ALL, False, tag=" [no bootstrap]")
    vs, pg = rl.rlcs_vtrace(g["rewards"], g["values"], g["log_rhos"], g["terminateds"],
                            with_pg=False)
    assert pg is None
    want = run_oracle("vtrace", src, dict(gamma=0.99, lambda_=1.0, rho_bar=1.0, c_bar=1.0), False)
    compare("vtrace", {"vs": vs}, {"vs": want["vs"]}, TOL)


@pytest.mark.parametrize("gamma,lam,rho_bar,c_bar", [(0.5, 0.5, 2.0, 0.5), (1.0, 1.0, 1.0, 1.0),
                                                     (0.0, 0.9, 1.0, 1.0), (0.9, 0.0, 0.3, 3.0)])
def test_hyperparameter_corners(rl, dev, gamma, lam, rho_bar, c_bar):
    src = rollout(6, 3000, 80, p_term=0.01, p_trunc=0.01)
    prm = dict(gamma=gamma, lambda_=lam, rho_bar=rho_bar, c_bar=c_bar)
    check_all(rl, src, to_dev(src, dev), prm, ALL, True, tag=" [%s]" % (prm,))


# --------------------------------------------------------------------------
# Workspace reuse, streams and graphs
# --------------------------------------------------------------------------

def test_workspace_reused_across_sizes(rl, dev):
    """The workspace self-resets: calls of different sizes and estimators on
    one stream, back to back, stay exact."""
    sizes = [(3, 5000), (40, 2100), (1, 70000), (3, 5000), (8, 9000)]
    srcs = [rollout(N, T, 90 + i, p_term=0.005) for i, (N, T) in enumerate(sizes)]
    gs = [to_dev(s, dev) for s in srcs]
    for rep in range(3):
        for src, g in zip(srcs, gs):
            for est in ("gae", "episodic_prefix_sum", "vtrace"):
                got = run_gpu(rl, est, g, DEFAULT, False)
                compare(est, got, run_oracle(est, src, DEFAULT, False), TOL)
    rl.check_all_workspaces()


def test_side_stream_gets_its_own_workspace(rl, dev):
    src = rollout(4, 30000, 95, p_term=0.001)
    g = to_dev(src, dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = {}
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs[s] = run_gpu(rl, "retrace", g, DEFAULT, False)
    torch.cuda.synchronize()
    want = run_oracle("retrace", src, DEFAULT, False)
    for s in (s1, s2):
        compare("retrace", outs[s], want, TOL)


def test_explicit_stream_argument_with_a_fresh_workspace(rl, dev):
    # stream= names a stream other than the current one; its first call
    # allocates and zeroes a workspace, which must be ordered on that stream
    src = rollout(4, 30000, 98, p_term=0.001)
    g = to_dev(src, dev)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    out = rl.rlcs_retrace(g["rewards"], g["values"], g["q_values"], g["log_rhos"],
                          g["terminateds"], DEFAULT["gamma"], DEFAULT["lambda_"],
                          DEFAULT["c_bar"], g["bootstrap_value"], stream=s)
    s.synchronize()
    compare("retrace", {"out": out}, run_oracle("retrace", src, DEFAULT, False), TOL)


def test_cuda_graph_capture_and_replay(rl, dev):
    src = rollout(16, 6000, 96, p_term=0.002, p_trunc=0.001)
    g = to_dev(src, dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):  # warm up: workspace allocated and zeroed outside capture
            run_gpu(rl, "vtrace", g, DEFAULT, True)
            run_gpu(rl, "episodic_prefix_sum", g, DEFAULT, False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        a = run_gpu(rl, "vtrace", g, DEFAULT, True)
        b = run_gpu(rl, "episodic_prefix_sum", g, DEFAULT, False)
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    compare("vtrace", a, run_oracle("vtrace", src, DEFAULT, True), TOL)
    compare("episodic_prefix_sum", b, run_oracle("episodic_prefix_sum", src, DEFAULT, False), TOL)
    rl.check_all_workspaces()


def test_outputs_are_deterministic_for_the_integer_path(rl, dev):
    src = rollout(2, 200000, 97, p_term=1e-4)
    g = to_dev(src, dev)
    first = run_gpu(rl, "episodic_prefix_sum", g, DEFAULT, False)["out"].clone()
    for _ in range(5):
        again = run_gpu(rl, "episodic_prefix_sum", g, DEFAULT, False)["out"]
        assert torch.equal(first, again)


@pytest.mark.parametrize("N,T", [(4096, 128), (64, 20000)])
@pytest.mark.parametrize("bars", [(1.0, 1.0), (5.0, 2.0)])
def test_extreme_ratios_and_magnitudes(rl, dev, N, T, bars):
    # log-ratios spread so far that exp overflows float (clipped to the bar)
    # or underflows (traces vanish and cut the carry); rewards and values of
    # magnitude 1e4. The oracle evaluates exp in double: overflow clips to
    # the same bar, underflow differs by less than 1e-38. Outputs are
    # compared in units of the input scale: vs = V + A cancels terms of
    # order 1e4, whose fp32 rounding no reordering avoids.
    scale = 1e4
    src = rollout(N, T, 99, p_term=0.01, p_trunc=0.005)
    rng = np.random.default_rng(7)
    src["log_rhos"] = (rng.standard_normal((N, T)) * 30.0).astype(np.float32)
    for k in ("rewards", "values", "q_values", "next_values", "bootstrap_value"):
        src[k] = (src[k] * scale).astype(np.float32)
    prm = dict(DEFAULT, rho_bar=bars[0], c_bar=bars[1])
    g = to_dev(src, dev)
    for est in ("vtrace", "retrace"):
        for trunc in (False, True):
            got = {k: v / scale for k, v in run_gpu(rl, est, g, prm, trunc).items()}
            want = {k: v / scale for k, v in run_oracle(est, src, prm, trunc).items()}
            compare(est, got, want, TOL, " [%dx%d %s]" % (N, T, bars))
    rl.check_all_workspaces()


def test_undamped_long_horizons(rl, dev):
    """lambda = 1 and gamma = 0.997 over 16384 steps: GAE, TD(lambda) returns
    and traces then have the horizon of discounted returns (about 333 steps
    with no damping), where rounding the multiplier's powers in fp32 would
    add up."""
    src = rollout(64, 16384, 6100, p_term=0.001, p_trunc=0.0005)
    prm = dict(gamma=0.997, lambda_=1.0, rho_bar=1.0, c_bar=1.0)
    check_all(rl, src, to_dev(src, dev), prm,
              ("gae", "lambda_returns", "discounted_returns", "eligibility_traces"), True,
              tag=" [undamped]")
