"""The launch planner, checked on the host (no GPU, no kernel launched).

rlcs_internal_plan runs the same planner as the entry points and reports
its choice: the launch shape, the tile (or chunk) length and how many of
them chain along a row, the warps per block and strips per warp, and whether
a block-tile grid spans more than one wave. Without a GPU the SM count is
taken as 152 (GB300's); the expectations below are written in terms of the
count the library reports, so they hold on any device.

The rules under test:
  * T <= 512: one warp per row, 1, 2 or 4 strips of 128 steps;
  * T <= 1024 and T <= 2048: one 1024- or 2048-step tile of 8 warps per
    row, so the row needs no look-back;
  * T <= 4096: one 4096-step tile of 16 warps of 2 strips per row;
  * longer rows: 8192-step tiles (32 warps of 2 strips) for T > 8192 while
    N * ceil(T / 8192) fits in one block per SM, else 4096-step tiles while
    N * ceil(T / 4096) fits in one wave of two blocks per SM, 2048-step
    tiles (8 warps of 2 strips) otherwise;
  * many_waves: N * tiles_per_row > 2 * SMs;
  * time-major: chunks of 128 steps of 32 environments, 16 warps of 8 steps
    below T = 1024 and 8 warps of 16 steps from there; with at most 256
    environments and T >= 2048, chunks of 8 environments: 1024 steps (16
    warps of 4 runs of 16 steps) when that grid fits in one block per SM,
    512 steps (8 warps) otherwise; their look-back reads four predecessors
    per warp and round for at most 16 groups of at least 16 chunks, else one.
"""
import ctypes

import pytest

from tests.test_boundary import INTERNAL, INVALID, OK

WARP_ROW, BLOCK_CHUNK, BLOCK_TILE, TIME_MAJOR = 1, 2, 3, 100


class PlanInfo(ctypes.Structure):
    _fields_ = [("shape", ctypes.c_int), ("sms", ctypes.c_int), ("tile", ctypes.c_int64),
                ("tiles_per_row", ctypes.c_int64), ("warps", ctypes.c_int),
                ("strips", ctypes.c_int), ("many_waves", ctypes.c_int), ("envs", ctypes.c_int),
                ("lookback_slots", ctypes.c_int)]


@pytest.fixture(scope="module")
def plan():
    import __graft_entry__
    __graft_entry__.build()
    from linear_recurrence_scan_affine_gb300 import binding
    c = binding.lib()
    c.rlcs_internal_plan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                     ctypes.POINTER(PlanInfo)]
    c.rlcs_internal_plan.restype = ctypes.c_int

    def run(N, T, time_major=False):
        info = PlanInfo()
        assert c.rlcs_internal_plan(N, T, int(time_major), ctypes.byref(info)) == OK
        return info
    run.lib = c
    return run


def test_the_header_struct_matches():
    src = open(INTERNAL).read()
    body = src[src.index("typedef struct {", src.index("RLCS_PLAN_TIME_MAJOR")):]
    body = body[:body.index("} rlcs_plan_info;")]
    fields = [ln.strip().rstrip(";").split()[-1] for ln in body.splitlines()[1:] if ln.strip()]
    assert fields == [f for f, _ in PlanInfo._fields_]


@pytest.mark.parametrize("T,strips", [(1, 1), (128, 1), (129, 2), (256, 2), (257, 4), (512, 4)])
def test_short_rows_take_one_warp_per_row(plan, T, strips):
    p = plan(4096, T)
    assert (p.shape, p.warps, p.strips, p.tile, p.tiles_per_row) == (WARP_ROW, 1, strips,
                                                                      128 * strips, 1)


@pytest.mark.parametrize("T,tile,warps,strips", [(513, 1024, 8, 1), (1024, 1024, 8, 1),
                                                 (1025, 2048, 8, 2), (2048, 2048, 8, 2),
                                                 (2049, 4096, 16, 2), (4096, 4096, 16, 2)])
@pytest.mark.parametrize("N", [1, 256, 4096, 100000])
def test_rows_up_to_4096_steps_are_one_tile(plan, N, T, tile, warps, strips):
    p = plan(N, T)
    assert (p.shape, p.tile, p.warps, p.strips, p.tiles_per_row) == (BLOCK_TILE, tile, warps,
                                                                      strips, 1)
    assert p.many_waves == int(N > 2 * p.sms)


@pytest.mark.parametrize("N,T", [(8, 131072), (64, 16384), (256, 8192), (256, 16384),
                                 (4096, 8192), (3, 10000), (300, 5000), (152, 8192),
                                 (153, 8192), (76, 16384), (77, 16385), (152, 8193)])
def test_longer_rows_chain_tiles(plan, N, T):
    p = plan(N, T)
    if T > 8192 and N * -(-T // 8192) <= p.sms:
        tile = 8192
    elif N * -(-T // 4096) <= 2 * p.sms:
        tile = 4096
    else:
        tile = 2048
    assert p.shape == BLOCK_TILE and p.tile == tile
    assert (p.warps, p.strips) == {8192: (32, 2), 4096: (16, 2), 2048: (8, 2)}[tile]
    assert p.tiles_per_row == -(-T // tile) and p.tiles_per_row > 1
    assert p.many_waves == int(N * p.tiles_per_row > 2 * p.sms)


def test_the_recipes(plan):
    # the long-row workloads on GB300 (152 SMs)
    p = plan(8, 131072)
    if p.sms == 152:
        assert (p.tile, p.warps, p.tiles_per_row, p.many_waves) == (8192, 32, 16, 0)
        p = plan(256, 16384)
        assert (p.tile, p.warps, p.tiles_per_row, p.many_waves) == (2048, 8, 8, 1)
        p = plan(256, 4096)
        assert (p.tile, p.warps, p.tiles_per_row, p.many_waves) == (4096, 16, 1, 0)
        p = plan(256, 1024)
        assert (p.tile, p.warps, p.tiles_per_row) == (1024, 8, 1)


@pytest.mark.parametrize("N,T,chunks,lane_steps", [(4096, 128, 1, 8), (7, 1, 1, 8),
                                                    (33, 129, 2, 8), (256, 1023, 8, 8),
                                                    (256, 1024, 8, 16), (257, 2048, 16, 16),
                                                    (4096, 4096, 32, 16), (256, 2047, 16, 16)])
def test_time_major_chunks(plan, N, T, chunks, lane_steps):
    p = plan(N, T, time_major=True)
    assert (p.shape, p.tile, p.tiles_per_row, p.strips, p.warps, p.envs) == (
        TIME_MAJOR, 128, chunks, lane_steps, 128 // lane_steps, 32)


@pytest.mark.parametrize("N,T", [(8, 131072), (1, 2048), (256, 2048), (256, 16384), (100, 5000),
                                 (128, 16384), (152, 8192)])
def test_time_major_few_environments_take_narrow_chunks(plan, N, T):
    p = plan(N, T, time_major=True)
    # 16 warps (1024-step chunks) when that grid fits in one block per SM
    wide = -(-N // 8) * -(-T // 1024) <= p.sms
    tile, warps = (1024, 16) if wide else (512, 8)
    assert (p.shape, p.tile, p.tiles_per_row, p.strips, p.warps, p.envs) == (
        TIME_MAJOR, tile, -(-T // tile), 16, warps, 8)
    if p.sms == 152:
        assert wide == ((N, T) not in ((256, 16384), (128, 16384)))


@pytest.mark.parametrize("N,T,slots", [(8, 131072, 4), (64, 16384, 4), (128, 16384, 4),
                                       (32, 65536, 4), (13, 20000, 4), (100, 40000, 4),
                                       (256, 16384, 1), (200, 20000, 1), (256, 4096, 1),
                                       (9, 4097, 1), (129, 16384, 1), (4096, 4096, 1)])
def test_time_major_lookback_window(plan, N, T, slots):
    # four predecessors per warp and round for few 8-environment groups
    # (at most 16) with long chains (at least 16 chunks); one otherwise, and
    # always one for the 32-environment chunks
    p = plan(N, T, time_major=True)
    if p.envs == 8:
        groups, chunks = -(-N // 8), p.tiles_per_row
        assert p.lookback_slots == (4 if groups <= 16 and chunks >= 16 else 1)
    else:
        assert p.lookback_slots == 1
    if p.sms == 152:
        assert p.lookback_slots == slots


def test_bad_arguments(plan):
    c, info = plan.lib, PlanInfo()
    assert c.rlcs_internal_plan(0, 128, 0, ctypes.byref(info)) == INVALID
    assert c.rlcs_internal_plan(4, 0, 0, ctypes.byref(info)) == INVALID
    assert c.rlcs_internal_plan(4, 128, 0, None) == INVALID


def test_refuses_while_a_shape_is_forced(plan):
    c, info = plan.lib, PlanInfo()
    assert c.rlcs_set_shape_override(BLOCK_TILE, 1024) == OK
    try:
        assert c.rlcs_internal_plan(4, 5000, 0, ctypes.byref(info)) == INVALID
    finally:
        assert c.rlcs_set_shape_override(0, 0) == OK
