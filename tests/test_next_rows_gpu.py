"""GPU parity for the two entry points beyond the seven estimators:

* rlcs_gae_and_returns: GAE and TD(lambda) returns from one pass, each
  checked against its own float64 oracle;
* rlcs_affine_scan: the recurrence on raw coefficients, forward and reverse,
  with and without resets and an initial value, against the affine oracle.

Same bar as the estimators: |gpu - oracle| <= 1e-4 * max(1, |oracle|)
(1e-3 at T = 131072). Every launch shape is forced on ragged sizes.
"""
import pytest
import torch

import oracle
from synthetic_rollouts import WORKLOADS, affine_inputs, rollout, workload_inputs
from tests.parity_common import TOL, TOL_VLONG, compare, params_of, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(0, 0), (1, 0), (2, 1024), (2, 4096), (3, 1024), (3, 2048), (3, 4096)]


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    yield rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def _fused(rl, src, g, prm, trunc, tol):
    tr = dict(truncateds=g["truncateds"], next_values=g["next_values"]) if trunc else {}
    trn = dict(truncateds=src["truncateds"], next_values=src["next_values"]) if trunc else {}
    adv, ret = rl.rlcs_gae_and_returns(g["rewards"], g["values"], g["terminateds"],
                                       prm["gamma"], prm["lambda_"], g["bootstrap_value"], **tr)
    compare("gae", {"out": adv}, {"out": oracle.gae(src["rewards"], src["values"],
            src["terminateds"], prm["gamma"], prm["lambda_"], src["bootstrap_value"], **trn)}, tol)
    compare("lambda_returns", {"out": ret}, {"out": oracle.lambda_returns(
        src["rewards"], src["values"], src["terminateds"], prm["gamma"], prm["lambda_"],
        src["bootstrap_value"], **trn)}, tol)
    rl.check_all_workspaces()


@pytest.mark.parametrize("name", ["gae_64x512", "all7_4096x128", "trunc5_4096x128",
                                  "longT_256x4096", "longT_256x16384"])
def test_gae_and_returns_workloads(rl, name):
    w = WORKLOADS[name]
    src = workload_inputs(w)
    _fused(rl, src, to_dev(src, torch.device("cuda:0")), params_of(w), w.p_trunc > 0, TOL)


@pytest.mark.parametrize("shape,chunk", SHAPES)
@pytest.mark.parametrize("T", [1, 127, 300, 2500, 9001])
def test_gae_and_returns_shapes(rl, shape, chunk, T):
    if shape == 1 and T > 512:
        pytest.skip("warp-row shape is for T <= 512")
    rl.rlcs_set_shape_override(shape, chunk)
    try:
        src = rollout(5, T, 6000 + T, p_term=0.01, p_trunc=0.005)
        _fused(rl, src, to_dev(src, torch.device("cuda:0")),
               dict(gamma=0.99, lambda_=0.95), True, TOL)
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def _affine(rl, N, T, seed, reverse, with_reset, with_init, tol=TOL, offset=0):
    src = affine_inputs(N, T, seed)
    g = to_dev(src, torch.device("cuda:0"), offset=offset)
    rs = g["reset"] if with_reset else None
    x0 = g["x_init"] if with_init else None
    got = rl.rlcs_affine_scan(g["a"], g["b"], rs, x0, reverse=reverse)
    want = oracle.affine_scan(src["a"], src["b"], src["reset"] if with_reset else None,
                              src["x_init"] if with_init else None, reverse=reverse)
    compare("affine_scan", {"out": got}, {"out": want}, tol)
    rl.check_all_workspaces()


@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("with_reset", [False, True])
@pytest.mark.parametrize("with_init", [False, True])
@pytest.mark.parametrize("N,T", [(4096, 128), (64, 512), (256, 4096), (256, 16384), (8, 131072)])
def test_affine_scan_sizes(rl, reverse, with_reset, with_init, N, T):
    _affine(rl, N, T, 7000 + T, reverse, with_reset, with_init, TOL_VLONG if T > 16384 else TOL)


@pytest.mark.parametrize("shape,chunk", SHAPES)
@pytest.mark.parametrize("T", [1, 5, 129, 512, 1025, 6000])
@pytest.mark.parametrize("reverse", [False, True])
def test_affine_scan_shapes(rl, shape, chunk, T, reverse):
    if shape == 1 and T > 512:
        pytest.skip("warp-row shape is for T <= 512")
    rl.rlcs_set_shape_override(shape, chunk)
    try:
        _affine(rl, 7, T, 8000 + T, reverse, True, True)
        _affine(rl, 3, T, 8100 + T, reverse, True, True, offset=1)   # unaligned rows
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


# --------------------------------------------------------------------------
# Compact input formats: bf16 rewards/values/next_values, uint8 masks
# --------------------------------------------------------------------------

def _compact(rl, N, T, seed, trunc, offset=0):
    from synthetic_rollouts import compact_rollout
    comp, f32 = compact_rollout(N, T, seed, p_term=0.01, p_trunc=0.005 if trunc else 0.0)
    g = to_dev(comp, torch.device("cuda:0"), offset=offset)
    kw = dict(truncateds=g["truncateds"], next_values=g["next_values"]) if trunc else {}
    got = rl.rlcs_gae_compact(g["rewards"], g["values"], g["terminateds"], 0.99, 0.95,
                              g["bootstrap_value"], **kw)
    kwn = dict(truncateds=f32["truncateds"], next_values=f32["next_values"]) if trunc else {}
    # the oracle sees exactly the values the compact arrays encode
    want = oracle.gae(f32["rewards"], f32["values"], f32["terminateds"], 0.99, 0.95,
                      f32["bootstrap_value"], **kwn)
    compare("gae", {"out": got}, {"out": want}, TOL)
    rl.check_all_workspaces()


@pytest.mark.parametrize("N,T", [(4096, 128), (64, 512), (256, 4096), (256, 16384)])
@pytest.mark.parametrize("trunc", [False, True])
def test_gae_compact_sizes(rl, N, T, trunc):
    _compact(rl, N, T, 9000 + T, trunc)


@pytest.mark.parametrize("N,T", [(1, 8), (300, 8), (37, 16), (33, 120), (7, 200), (300, 1000),
                                 (5, 2040), (19, 2048), (3, 2056), (3, 3000), (400, 4096),
                                 (41, 6000), (9, 8200), (2, 20000), (300, 6000), (20000, 128),
                                 (37, 132), (9, 1028), (3, 1024), (700, 512), (13000, 256), (76, 16384)])
@pytest.mark.parametrize("trunc", [False, True])
def test_gae_compact_eight_step_tiles(rl, N, T, trunc):
    """The automatic shape for T % 8 == 0: whole rows packed into tiles of
    8 warps (2048 steps, T <= 2048) or 16 warps (4096 steps, T <= 4096),
    with a ragged last tile, rows of 8 steps and rows that fill a tile;
    chained tiles beyond (ragged last tile per row); both register budgets
    (one-wave and larger grids). T % 8 != 0 and unaligned arrays take the
    other shapes."""
    _compact(rl, N, T, 9300 + N + T, trunc)
    _compact(rl, N, T, 9400 + N + T, trunc, offset=1)


@pytest.mark.parametrize("shape,chunk", SHAPES)
@pytest.mark.parametrize("T", [1, 3, 130, 511, 2049, 7000])
def test_gae_compact_shapes(rl, shape, chunk, T):
    if shape == 1 and T > 512:
        pytest.skip("warp-row shape is for T <= 512")
    rl.rlcs_set_shape_override(shape, chunk)
    try:
        _compact(rl, 5, T, 9100 + T, True)
        _compact(rl, 3, T, 9200 + T, True, offset=1)   # unaligned rows: scalar loads
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def test_diag_stream_copy_sums_inputs(rl):
    dev = torch.device("cuda:0")
    ins = [torch.randn(64, 256, device=dev) for _ in range(3)]
    out = torch.empty(64, 256, device=dev)
    rl.rlcs_diag_stream_copy(ins, out)
    torch.cuda.synchronize()
    assert torch.allclose(out, ins[0] + ins[1] + ins[2], rtol=0, atol=1e-6)
    out.fill_(7.0)
    rl.rlcs_diag_stream_copy(ins, out, empty=True)   # only waits: leaves out alone
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
