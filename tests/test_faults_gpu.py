"""Failure detection without a GPU fault.

Every device-side wait in the library is bounded: on expiry the kernel records
RLCS_ERR_TIMEOUT in the workspace status word and finishes, so the context
stays usable. These tests make a look-back wait run out on purpose by
corrupting the workspace on the host: for the ticket-ordered chunk shape its
ticket counter starts at 1, so chunk ticket 0 is never handed out and its
successor waits for a flag that nothing sets; for the time-major shape the
epoch moves in mid-launch (see that test). Each checks that the call returns,
that rlcs_check_status reports the timeout, and that after
rlcs_workspace_init the next call is correct again. Nothing here traps,
faults or hangs the GPU: a wait gives up after about a second.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from synthetic_rollouts import rollout
from tests.parity_common import TOL, compare, run_oracle

pytestmark = pytest.mark.gpu

RLCS_OK, RLCS_ERR_TIMEOUT = 0, 5


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_bounded_lookback_wait_reports_timeout_and_recovers():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    c = rl.lib()
    dev = torch.device("cuda:0")
    N, T = 1, 4096
    src = rollout(N, T, 777, p_term=0.002)
    g = {k: torch.from_numpy(v).to(dev) for k, v in src.items()}
    out = torch.empty_like(g["rewards"])
    nbytes = c.rlcs_workspace_bytes(N, T)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    prm = dict(gamma=0.99, lambda_=0.95, rho_bar=1.0, c_bar=1.0)
    want = run_oracle("gae", src, prm, False)

    def call():
        return c.rlcs_gae(_p(g["rewards"]), _p(g["values"]), _p(g["terminateds"]), None, None,
                          _p(g["bootstrap_value"]), _p(out), N, T, 0.99, 0.95, _p(ws), nbytes,
                          stream)

    # ticket-ordered chunks of 1024 steps: four chunks, three of them wait
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_BLOCK_CHUNK, 1024)
    try:
        assert call() == RLCS_OK
        assert c.rlcs_check_status(_p(ws), stream) == RLCS_OK
        compare("gae", {"out": out}, want, TOL)

        ws.view(torch.int32)[1] = 1  # header word 1: next chunk ticket
        t0 = time.perf_counter()
        assert call() == RLCS_OK     # the launch itself is fine
        status = c.rlcs_check_status(_p(ws), stream)  # synchronises
        elapsed = time.perf_counter() - t0
        assert status == RLCS_ERR_TIMEOUT, c.rlcs_status_string(status)
        assert 0.5 < elapsed < 30.0, elapsed
        # the status word is cleared by reading it
        assert c.rlcs_check_status(_p(ws), stream) == RLCS_OK

        assert c.rlcs_workspace_init(_p(ws), nbytes, stream) == RLCS_OK
        out.fill_(float("nan"))
        assert call() == RLCS_OK
        assert c.rlcs_check_status(_p(ws), stream) == RLCS_OK
        compare("gae", {"out": out}, want, TOL)
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def test_time_major_lookback_wait_reports_timeout_and_recovers():
    # The time-major chain has no ticket: chunk order is the block order. Its
    # epoch is what a host-side corruption can break. Presetting the
    # finished-block counter to its last value makes the first block that
    # finishes move the workspace to the next epoch in mid-launch; the first
    # block dispatched after that waits on a predecessor whose records carry
    # the old epoch's tag, which never matches, so its bounded wait runs out.
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    c = rl.lib()
    dev = torch.device("cuda:0")
    N, T = 32, 1 << 18  # thousands of chunks: more blocks than fit on the GPU at once
    src = rollout(N, T, 778, p_term=0.002)
    g = {k: (torch.from_numpy(np.ascontiguousarray(v.T)).to(dev) if v.ndim == 2
             else torch.from_numpy(v).to(dev)) for k, v in src.items()}
    out = torch.empty_like(g["rewards"])
    nbytes = c.rlcs_workspace_bytes_tm(N, T)
    blocks = (nbytes - 64) // 32 // 32  # one 32-byte record per lane, 32 lanes a block
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    want = run_oracle("gae", src, dict(gamma=0.99, lambda_=0.95, rho_bar=1.0, c_bar=1.0), False)

    def call():
        return c.rlcs_gae_tm(_p(g["rewards"]), _p(g["values"]), _p(g["terminateds"]), None, None,
                             _p(g["bootstrap_value"]), _p(out), N, T, 0.99, 0.95, _p(ws), nbytes,
                             stream)

    def check():
        compare("gae", {"out": out.cpu().numpy().T}, want, TOL)

    assert call() == RLCS_OK
    assert c.rlcs_check_status(_p(ws), stream) == RLCS_OK
    check()

    ws.view(torch.int32)[2] = blocks - 1  # header word 2: blocks finished
    t0 = time.perf_counter()
    assert call() == RLCS_OK
    status = c.rlcs_check_status(_p(ws), stream)
    elapsed = time.perf_counter() - t0
    assert status == RLCS_ERR_TIMEOUT, c.rlcs_status_string(status)
    assert 0.5 < elapsed < 30.0, elapsed

    assert c.rlcs_workspace_init(_p(ws), nbytes, stream) == RLCS_OK
    out.fill_(float("nan"))
    assert call() == RLCS_OK
    assert c.rlcs_check_status(_p(ws), stream) == RLCS_OK
    check()
