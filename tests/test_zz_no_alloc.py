"""rlcs_gae_noalloc: GAE for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all (a plugin inside a host program
that owns every device allocation, a real-time loop that forbids allocating
after start-up), so they cannot provide the workspace that long rows need.
rlcs_gae_noalloc takes no workspace; its scratch is a fixed array inside the
library. These tests call it through the C ABI and check two calls in a row
against the float64 oracle, element by element, within the parity tolerance:
on long rows that chain many chunks through the scratch, on a mid-size case
and on short rows that need no scratch; a ticket-ordered chunk launch right
after a tile launch (the two shapes use the array's header differently); a
size beyond the array's capacity is refused before anything runs; and
rlcs_gae_noalloc_recover reports a wait that ran out and repairs the array.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes
import time

import pytest
import torch

from synthetic_rollouts import rollout
from tests.parity_common import TOL, TOL_VLONG, compare, run_oracle

pytestmark = pytest.mark.gpu

RLCS_OK, RLCS_ERR_WORKSPACE, RLCS_ERR_TIMEOUT = 0, 3, 5
GAMMA, LAMBDA = 0.99, 0.95
PRM = dict(gamma=GAMMA, lambda_=LAMBDA, rho_bar=1.0, c_bar=1.0)


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    import linear_recurrence_scan_affine_gb300 as rl
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    c = rl.lib()
    P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    c.rlcs_gae_noalloc.argtypes = [P] * 7 + [I64, I64, F, F, P]
    c.rlcs_gae_noalloc.restype = ctypes.c_int
    c.rlcs_gae_noalloc_recover.argtypes = [P]
    c.rlcs_gae_noalloc_recover.restype = ctypes.c_int
    c.rlcs_internal_noalloc_scratch.argtypes = [ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]
    c.rlcs_internal_noalloc_scratch.restype = ctypes.c_int
    yield rl, c
    rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


class _Case:
    """One seeded rollout on the device, its oracle result and a noalloc call."""

    def __init__(self, N, T, seed, trunc):
        self.N, self.T, self.trunc = N, T, trunc
        self.src = rollout(N, T, seed, p_term=1e-3, p_trunc=5e-4 if trunc else 0.0)
        dev = torch.device("cuda:0")
        self.g = {k: torch.from_numpy(v).to(dev) for k, v in self.src.items()}
        self.want = run_oracle("gae", self.src, PRM, trunc)
        self.tol = TOL if T <= 16384 else TOL_VLONG

    def call(self, c, out):
        g = self.g
        tr, nv = (g["truncateds"], g["next_values"]) if self.trunc else (None, None)
        return c.rlcs_gae_noalloc(_p(g["rewards"]), _p(g["values"]), _p(g["terminateds"]),
                                  _p(tr), _p(nv), _p(g["bootstrap_value"]), _p(out), self.N,
                                  self.T, GAMMA, LAMBDA, _stream())

    def check(self, c, tag):
        out = torch.full_like(self.g["rewards"], float("nan"))
        st = self.call(c, out)
        assert st == RLCS_OK, c.rlcs_status_string(st)
        torch.cuda.synchronize()
        compare("gae", {"out": out}, self.want, self.tol, tag)


@pytest.mark.parametrize("N,T,trunc", [(8, 131072, True), (256, 4096, False), (4096, 128, True)])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(lib, N, T, trunc):
    rl, c = lib
    case = _Case(N, T, 4242 + T, trunc)
    for call in range(2):
        case.check(c, " (noalloc call %d)" % call)
    assert c.rlcs_gae_noalloc_recover(_stream()) == RLCS_OK


def test_noalloc_chunk_shape_after_tile_shape(lib):
    # The default tile shape orders blocks by index and leaves the header's
    # ticket counter alone; the chunk shape draws tickets from it. A chunk
    # launch right after tile launches must find it at zero, and a tile
    # launch after that must still find the epoch moving.
    rl, c = lib
    case = _Case(3, 10000, 5151, True)
    try:
        case.check(c, " (tile shape)")
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_BLOCK_CHUNK, 1024)
        case.check(c, " (chunk shape, first)")
        case.check(c, " (chunk shape, second)")
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)
    case.check(c, " (tile shape again)")
    assert c.rlcs_gae_noalloc_recover(_stream()) == RLCS_OK


class _DeviceWords:
    """A device array the library owns, seen as uint32 words by torch."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<u4", "data": (ptr, False),
                                         "version": 3}


def test_noalloc_recover_reports_a_timeout_and_repairs_the_array(lib):
    # Host-side fault injection, as for the caller-workspace entry points:
    # the scratch header's ticket counter is set to 1, so the ticket-ordered
    # chunk shape never hands out chunk 0 and its successor's bounded wait
    # runs out after about a second. No GPU fault is involved.
    rl, c = lib
    ptr, size = ctypes.c_void_p(), ctypes.c_size_t()
    assert c.rlcs_internal_noalloc_scratch(ctypes.byref(ptr), ctypes.byref(size)) == RLCS_OK
    assert ptr.value and size.value >= 64
    header = torch.as_tensor(_DeviceWords(ptr.value, 16), device="cuda:0")
    case = _Case(1, 4096, 6161, False)
    try:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_BLOCK_CHUNK, 1024)
        case.check(c, " (before the fault)")
        assert c.rlcs_gae_noalloc_recover(_stream()) == RLCS_OK

        header[1] = 1  # word 1: the next chunk ticket
        torch.cuda.synchronize()
        out = torch.empty_like(case.g["rewards"])
        t0 = time.perf_counter()
        assert case.call(c, out) == RLCS_OK  # the launch itself is fine
        status = c.rlcs_gae_noalloc_recover(_stream())
        elapsed = time.perf_counter() - t0
        assert status == RLCS_ERR_TIMEOUT, c.rlcs_status_string(status)
        assert 0.5 < elapsed < 30.0, elapsed
        assert int(header.sum().item()) == 0  # the header is zeroed again

        for call in range(2):
            case.check(c, " (after recovery, call %d)" % call)
        assert c.rlcs_gae_noalloc_recover(_stream()) == RLCS_OK
    finally:
        rl.rlcs_set_shape_override(rl.RLCS_SHAPE_AUTO, 0)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    rl, c = lib
    fake = [ctypes.c_void_p(0x7f0000000000 + i * (1 << 36)) for i in range(4)]
    # 65537 rows of 1024 steps need 65537 chunk records; the array holds 65536
    st = c.rlcs_gae_noalloc(fake[0], fake[1], fake[2], None, None, None, fake[3], 65537, 1024,
                            GAMMA, LAMBDA, None)
    assert st == RLCS_ERR_WORKSPACE
