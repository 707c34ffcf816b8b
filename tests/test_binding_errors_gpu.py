"""The Python binding's argument handling on CUDA tensors.

Every rejected call here is refused on the host before anything launches:
shape, dtype and device errors in the binding (ValueError / TypeError), and
the C ABI's own checks (RlcsError with the status the header documents) for
empty batches, a truncation mask without its next values, and outputs that
overlap an input or each other. Accepted corner forms (a 1-D row, a
non-contiguous input) are checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from synthetic_rollouts import rollout
from tests.parity_common import TOL, compare

pytestmark = pytest.mark.gpu

INVALID_ARG = 1


@pytest.fixture(scope="module")
def rl():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    return rl


@pytest.fixture(scope="module")
def g():
    src = rollout(6, 300, 9500, p_term=0.02, p_trunc=0.01)
    return {k: torch.from_numpy(v).cuda() for k, v in src.items()}, src


@pytest.mark.parametrize("shape", [(0, 128), (4, 0), (0, 0)])
def test_empty_batches_are_invalid(rl, shape):
    z = torch.zeros(shape, device="cuda")
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_gae(z, z.clone(), z.clone(), 0.99, 0.95)
    assert e.value.status == INVALID_ARG
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_episodic_prefix_sum(torch.zeros(shape, dtype=torch.int32, device="cuda"), z)
    assert e.value.status == INVALID_ARG
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_gae_tm(z, z.clone(), z.clone(), 0.99, 0.95)
    assert e.value.status == INVALID_ARG


def test_shape_dtype_and_device_errors(rl, g):
    d, _ = g
    r, v, t = d["rewards"], d["values"], d["terminateds"]
    with pytest.raises(ValueError):
        rl.rlcs_gae(r, v[:, :-4], t)                       # values shorter than rewards
    with pytest.raises(TypeError):
        rl.rlcs_gae(r, v.double(), t)                      # float64 values
    with pytest.raises(ValueError):
        rl.rlcs_gae(r.cpu(), v, t)                          # host tensor
    with pytest.raises(ValueError):
        rl.rlcs_gae(r, v, t, bootstrap_value=d["bootstrap_value"][:-1])
    with pytest.raises(ValueError):
        rl.rlcs_gae(r.reshape(2, 3, 300), v, t)            # not [N, T]
    with pytest.raises(TypeError):
        rl.rlcs_episodic_prefix_sum(d["x"], t)              # prefix sum takes int32
    with pytest.raises(ValueError):
        rl.rlcs_gae(r, v, t, truncateds=d["truncateds"][:, :-4],
                    next_values=d["next_values"][:, :-4])


def test_truncation_mask_without_next_values_is_invalid(rl, g):
    d, _ = g
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_gae(d["rewards"], d["values"], d["terminateds"], truncateds=d["truncateds"])
    assert e.value.status == INVALID_ARG
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_vtrace(d["rewards"], d["values"], d["log_rhos"], d["terminateds"],
                       next_values=d["next_values"])
    assert e.value.status == INVALID_ARG


def test_outputs_overlapping_inputs_are_invalid(rl, g):
    d, _ = g
    r = d["rewards"].clone()
    v = d["values"].clone()
    with pytest.raises(rl.RlcsError) as e:
        rl.rlcs_gae(r, v, d["terminateds"], out=r)          # in place over rewards
    assert e.value.status == INVALID_ARG
    with pytest.raises(rl.RlcsError) as e:                   # overlapping by one row
        big = torch.empty(7, 300, device="cuda")
        big[:6] = v
        rl.rlcs_gae(r, big[:6], d["terminateds"], out=big[1:])
    assert e.value.status == INVALID_ARG
    vs = torch.empty_like(r)
    with pytest.raises(rl.RlcsError) as e:                   # vs and pg in one buffer
        rl.rlcs_vtrace(r, v, d["log_rhos"], d["terminateds"], out=vs, out_pg=vs)
    assert e.value.status == INVALID_ARG
    with pytest.raises(rl.RlcsError) as e:                   # output over the bootstrap values
        boot = torch.empty(6 * 300, device="cuda")
        boot[:6] = d["bootstrap_value"]
        rl.rlcs_discounted_returns(r, d["terminateds"], 0.99, boot[:6],
                                   out=boot.view(6, 300))
    assert e.value.status == INVALID_ARG
    # nothing was written by the refused calls
    assert torch.equal(r, d["rewards"]) and torch.equal(v, d["values"])


def test_one_dimensional_row_and_non_contiguous_inputs(rl, g):
    d, src = g
    got = rl.rlcs_gae(d["rewards"][2], d["values"][2], d["terminateds"][2], 0.99, 0.95)
    assert got.shape == (300,)
    want = oracle.gae(src["rewards"][2:3], src["values"][2:3], src["terminateds"][2:3],
                          0.99, 0.95)
    compare("gae", {"out": got.reshape(1, 300)}, {"out": want}, TOL)
    # a transposed view is made contiguous by the binding before the call
    rt = d["rewards"].T.contiguous().T
    vt = d["values"].T.contiguous().T
    assert not rt.is_contiguous()
    got = rl.rlcs_gae(rt, vt, d["terminateds"], 0.99, 0.95, d["bootstrap_value"])
    want = oracle.gae(src["rewards"], src["values"], src["terminateds"], 0.99, 0.95,
                          src["bootstrap_value"])
    compare("gae", {"out": got}, {"out": want}, TOL)
    assert np.isfinite(got.cpu().numpy()).all()


def test_caller_outputs_are_checked_before_the_call(rl, g):
    d, _ = g
    r, v, t = d["rewards"], d["values"], d["terminateds"]
    with pytest.raises(ValueError):                          # too few elements
        rl.rlcs_gae(r, v, t, out=torch.empty(5, 300, device="cuda"))
    with pytest.raises(TypeError):                           # wrong dtype
        rl.rlcs_gae(r, v, t, out=torch.empty(6, 300, dtype=torch.float64, device="cuda"))
    with pytest.raises(ValueError):                          # not contiguous
        rl.rlcs_gae(r, v, t, out=torch.empty(300, 6, device="cuda").T)
    with pytest.raises(ValueError):                          # host memory
        rl.rlcs_gae(r, v, t, out=torch.empty(6, 300))
    with pytest.raises(ValueError):
        rl.rlcs_vtrace(r, v, d["log_rhos"], t, out_pg=torch.empty(6, 299, device="cuda"))
    with pytest.raises(ValueError):
        rl.rlcs_gae_and_returns(r, v, t, out_returns=torch.empty(3, 300, device="cuda"))
    with pytest.raises(TypeError):                           # the prefix sum writes int32
        rl.rlcs_episodic_prefix_sum(d["x_int"], t, out=torch.empty(6, 300, device="cuda"))
    with pytest.raises(ValueError):
        rl.rlcs_gae_tm(r.T.contiguous(), v.T.contiguous(), t.T.contiguous(),
                       out=torch.empty(300, 5, device="cuda"))
    with pytest.raises(ValueError):
        rl.rlcs_run_group([("gae", dict(rewards=r, values=v, terminateds=t,
                                        out=torch.empty(6, 100, device="cuda")))])
    with pytest.raises(ValueError):
        rl.rlcs_diag_stream_copy([r, v[:, :200]], torch.empty(6, 300, device="cuda"))
    # a correct caller-provided output of another shape but the same elements is used as is
    o = torch.full((300 * 6,), float("nan"), device="cuda")
    got = rl.rlcs_gae(r, v, t, 0.99, 0.95, out=o)
    assert got.data_ptr() == o.data_ptr() and got.shape == (6, 300)
    assert torch.isfinite(o).all()
