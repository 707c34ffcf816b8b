"""rlcs_gae_noalloc: GAE for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all (a plugin inside a host program
that owns every device allocation, a real-time loop that forbids allocating
after start-up), so they cannot provide the workspace that long rows need.
rlcs_gae_noalloc takes no workspace; its scratch is a fixed array inside the
library. These tests call it through the C ABI and check that two calls in a
row match rlcs_gae (the entry point with a caller workspace) within the
parity tolerance: on long rows that chain many chunks through the scratch,
on a mid-size case, and on short rows that need no scratch. They also check
that a size beyond the array's capacity is refused before anything runs.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from synthetic_rollouts import rollout

pytestmark = pytest.mark.gpu

TOL = 1e-4
RLCS_OK, RLCS_ERR_WORKSPACE = 0, 3


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    c = rl.lib()
    P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    c.rlcs_gae_noalloc.argtypes = [P] * 7 + [I64, I64, F, F, P]
    c.rlcs_gae_noalloc.restype = ctypes.c_int
    return rl, c


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("N,T,trunc", [(8, 131072, True), (256, 4096, False), (4096, 128, True)])
def test_noalloc_matches_workspace_entry_point_twice(lib, N, T, trunc):
    rl, c = lib
    dev = torch.device("cuda:0")
    src = rollout(N, T, 4242 + T, p_term=1e-3, p_trunc=5e-4 if trunc else 0.0)
    g = {k: torch.from_numpy(v).to(dev) for k, v in src.items()}
    tr, nv = (g["truncateds"], g["next_values"]) if trunc else (None, None)
    ref = rl.rlcs_gae(g["rewards"], g["values"], g["terminateds"], 0.99, 0.95,
                      g["bootstrap_value"], truncateds=tr, next_values=nv)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(g["rewards"], float("nan"))
        st = c.rlcs_gae_noalloc(_p(g["rewards"]), _p(g["values"]), _p(g["terminateds"]), _p(tr),
                                _p(nv), _p(g["bootstrap_value"]), _p(out), N, T, 0.99, 0.95,
                                stream)
        assert st == RLCS_OK, c.rlcs_status_string(st)
        torch.cuda.synchronize()
        a, b = out.double().cpu().numpy(), ref.double().cpu().numpy()
        err = np.abs(a - b) / np.maximum(1.0, np.abs(b))
        assert np.all(np.isfinite(a)), "call %d: non-finite output" % call
        assert err.max() <= TOL, "call %d: max scaled error %.3g" % (call, err.max())


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    rl, c = lib
    fake = [ctypes.c_void_p(0x7f0000000000 + i * (1 << 36)) for i in range(4)]
    # 65537 rows of 1024 steps need 65537 chunk records; the array holds 65536
    st = c.rlcs_gae_noalloc(fake[0], fake[1], fake[2], None, None, None, fake[3], 65537, 1024,
                            0.99, 0.95, None)
    assert st == RLCS_ERR_WORKSPACE
