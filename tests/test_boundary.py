"""Host-side checks of the C ABI boundary (no GPU needed, no kernel launched).

The library must load, export every function include/rlcs.h declares, and
reject bad arguments with the documented status before anything reaches the
GPU. Fake device addresses are fine here: argument errors return before any
CUDA call that would touch them.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlcs.h")
INTERNAL = os.path.join(ROOT, "include", "rlcs_internal.h")

OK, INVALID, MISALIGNED, WORKSPACE, CUDA, TIMEOUT = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from linear_recurrence_scan_affine_gb300 import binding
    return binding.lib()


def declared_functions(path=None):
    """Functions the headers declare (both, unless one path is given)."""
    names = set()
    for p in ([path] if path else [HEADER, INTERNAL]):
        src = re.sub(r"/\*.*?\*/", "", open(p).read(), flags=re.S)
        names |= set(re.findall(r"\b(rlcs_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_test_hooks_live_outside_the_product_header():
    product = declared_functions(HEADER)
    internal = declared_functions(INTERNAL)
    for name in ("rlcs_set_shape_override", "rlcs_diag_stream_copy",
                 "rlcs_internal_noalloc_scratch", "rlcs_internal_plan"):
        assert name in internal and name not in product, name
    assert "rlcs_gae_noalloc" in product and "rlcs_gae_noalloc_recover" in product


def test_header_declares_the_seven_estimators():
    names = declared_functions()
    for est in ("gae", "vtrace", "retrace", "lambda_returns", "discounted_returns",
                "eligibility_traces", "episodic_prefix_sum"):
        assert "rlcs_" + est in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_match_nm():
    # the dynamic symbol table holds each declared function with C linkage
    import subprocess
    from linear_recurrence_scan_affine_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for name in declared_functions():
        assert name in syms, name


def test_status_strings(lib):
    for code in range(6):
        s = lib.rlcs_status_string(code).decode()
        assert s.startswith("RLCS_")
    assert lib.rlcs_status_string(99).decode() == "unknown rlcs_status"


def test_workspace_bytes(lib):
    assert lib.rlcs_workspace_bytes(0, 10) == 0
    assert lib.rlcs_workspace_bytes(10, 0) == 0
    assert lib.rlcs_workspace_bytes(-1, 10) == 0
    # 64-byte header + 32 bytes per 1024-step chunk of every row
    assert lib.rlcs_workspace_bytes(4096, 128) == 64 + 32 * 4096
    assert lib.rlcs_workspace_bytes(8, 131072) == 64 + 32 * 8 * 128
    assert lib.rlcs_workspace_bytes(3, 1025) == 64 + 32 * 3 * 2


FAKE = 0x7f0000000000  # 16-byte aligned fake device address, never dereferenced


def fake(i, nbytes=1 << 24):
    return ctypes.c_void_p(FAKE + i * nbytes)


def gae(lib, r, v, d, tr, nv, b, out, N, T, ws=None, wsb=0):
    return lib.rlcs_gae(r, v, d, tr, nv, b, out, N, T, 0.99, 0.95, ws, wsb, None)


def test_gae_rejects_bad_sizes(lib):
    a = [fake(i) for i in range(4)]
    for N, T in [(0, 8), (8, 0), (-1, 8), (8, -5), (1 << 40, 1 << 40)]:
        assert gae(lib, a[0], a[1], a[2], None, None, None, a[3], N, T) == INVALID


def test_rejects_null_required_pointers(lib):
    a = [fake(i) for i in range(4)]
    assert gae(lib, None, a[1], a[2], None, None, None, a[3], 4, 8) == INVALID
    assert gae(lib, a[0], None, a[2], None, None, None, a[3], 4, 8) == INVALID
    assert gae(lib, a[0], a[1], None, None, None, None, a[3], 4, 8) == INVALID
    assert gae(lib, a[0], a[1], a[2], None, None, None, None, 4, 8) == INVALID
    assert lib.rlcs_vtrace(a[0], a[1], None, a[2], None, None, None, a[3], None, 4, 8,
                           0.99, 1.0, 1.0, 1.0, None, 0, None) == INVALID
    assert lib.rlcs_retrace(a[0], a[1], a[2], None, a[3], None, None, None, fake(9), 4, 8,
                            0.99, 1.0, 1.0, None, 0, None) == INVALID
    assert lib.rlcs_eligibility_traces(None, a[1], a[2], 4, 8, 0.9, 0.9, None, 0, None) == INVALID
    assert lib.rlcs_episodic_prefix_sum(a[0], None, a[2], 4, 8, None, 0, None) == INVALID
    assert lib.rlcs_discounted_returns(a[0], a[1], None, None, None, None, 4, 8, 0.9,
                                       None, 0, None) == INVALID


def test_rejects_half_truncation_pair(lib):
    a = [fake(i) for i in range(6)]
    assert gae(lib, a[0], a[1], a[2], a[4], None, None, a[3], 4, 8) == INVALID
    assert gae(lib, a[0], a[1], a[2], None, a[5], None, a[3], 4, 8) == INVALID


def test_rejects_aliasing(lib):
    a = [fake(i) for i in range(4)]
    # output identical to an input
    assert gae(lib, a[0], a[1], a[2], None, None, None, a[0], 4, 8) == INVALID
    assert gae(lib, a[0], a[1], a[2], None, None, None, a[2], 4, 8) == INVALID
    # output overlapping an input by part of a row
    inner = ctypes.c_void_p(a[1].value + 16)
    assert gae(lib, a[0], a[1], a[2], None, None, None, inner, 4, 8) == INVALID
    # V-trace outputs overlapping each other
    assert lib.rlcs_vtrace(a[0], a[1], a[2], a[3], None, None, None, fake(7),
                           ctypes.c_void_p(fake(7).value + 64), 4, 8, 0.99, 1.0, 1.0, 1.0,
                           None, 0, None) == INVALID
    # output overlapping the bootstrap array
    assert gae(lib, a[0], a[1], a[2], None, None, fake(5), fake(5), 4, 8) == INVALID


def test_long_rows_need_a_workspace(lib):
    a = [fake(i, 1 << 30) for i in range(4)]
    lib.rlcs_set_shape_override(0, 0)
    N, T = 4, 1 << 16
    assert gae(lib, a[0], a[1], a[2], None, None, None, a[3], N, T) == WORKSPACE
    small = lib.rlcs_workspace_bytes(N, T) // 8
    assert gae(lib, a[0], a[1], a[2], None, None, None, a[3], N, T, fake(20, 1 << 30),
               small) == WORKSPACE


def test_time_major_workspace(lib):
    # one 32-byte record per environment (rounded up to groups of 32) and
    # chunk, after the 64-byte header; nonzero even when one chunk covers T
    assert lib.rlcs_workspace_bytes_tm(0, 10) == 0
    assert lib.rlcs_workspace_bytes_tm(10, 0) == 0
    one = lib.rlcs_workspace_bytes_tm(32, 1)
    assert one == 64 + 32 * 32
    assert lib.rlcs_workspace_bytes_tm(1, 1) == one
    per_chunk = 32 * 32
    chunk = next(t for t in range(1, 4097) if lib.rlcs_workspace_bytes_tm(32, t + 1) > one)
    assert chunk in (32, 64, 128, 256)
    assert lib.rlcs_workspace_bytes_tm(33, 3 * chunk) == 64 + 2 * 3 * per_chunk
    # rows longer than one chunk need it; a missing or short one launches nothing
    a = [fake(i) for i in range(4)]
    N, T = 4, 1000
    assert lib.rlcs_gae_tm(a[0], a[1], a[2], None, None, None, a[3], N, T, 0.99, 0.95, None, 0,
                           None) == WORKSPACE
    short = lib.rlcs_workspace_bytes_tm(N, T) - 32
    assert lib.rlcs_gae_tm(a[0], a[1], a[2], None, None, None, a[3], N, T, 0.99, 0.95, fake(9),
                           short, None) == WORKSPACE
    assert lib.rlcs_affine_scan_tm(a[0], a[1], None, None, a[3], N, T, 1, None, 0,
                                   None) == WORKSPACE


def test_shape_override_validation(lib):
    assert lib.rlcs_set_shape_override(7, 0) == INVALID
    assert lib.rlcs_set_shape_override(3, 512) == INVALID
    assert lib.rlcs_set_shape_override(3, 4096) == OK
    assert lib.rlcs_set_shape_override(2, 3000) == INVALID
    assert lib.rlcs_set_shape_override(2, 2048) == OK
    assert lib.rlcs_set_shape_override(3, 8192) == OK       # register tiles only
    assert lib.rlcs_set_shape_override(2, 8192) == INVALID
    assert lib.rlcs_set_shape_override(0, 0) == OK
    # warp-row is limited to T <= 512
    assert lib.rlcs_set_shape_override(1, 0) == OK
    a = [fake(i) for i in range(4)]
    assert gae(lib, a[0], a[1], a[2], None, None, None, a[3], 4, 1000) == INVALID
    assert lib.rlcs_set_shape_override(0, 0) == OK


def test_workspace_init_rejects_null(lib):
    assert lib.rlcs_workspace_init(None, 64, None) == INVALID


def test_compact_overlap_uses_element_sizes(lib):
    # A uint8 mask plane of N*T bytes ends before an output placed right after
    # it, although N*T float32 elements would reach into it. The rows are long
    # and no workspace is given, so a call that passes the overlap check stops
    # at the workspace check: nothing is ever launched on these fake pointers.
    N, T = 4, 16384                                 # four 4096-step tiles per row
    r, v, d = fake(0), fake(1), fake(2)
    out = ctypes.c_void_p(d.value + N * T)          # right after the uint8 masks
    assert lib.rlcs_gae_compact(r, v, d, None, None, None, out, N, T, 0.99, 0.95, None, 0,
                                None) == WORKSPACE
    inside = ctypes.c_void_p(d.value + N * T - 16)  # overlapping the masks
    assert lib.rlcs_gae_compact(r, v, d, None, None, None, inside, N, T, 0.99, 0.95, None, 0,
                                None) == INVALID


def test_rlcs_call_layout_matches_the_header(tmp_path):
    # the ctypes mirror of rlcs_call has the C struct's size and offsets
    import ctypes as ct
    import subprocess
    from linear_recurrence_scan_affine_gb300.binding import RlcsCall
    fields = [f for f, _ in RlcsCall._fields_]
    cname = {"lambda_": "lambda"}
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "rlcs.h"\nint main(void) {\n'
                    '  printf("%zu\\n", sizeof(rlcs_call));\n'
                    + "".join('  printf("%%zu\\n", offsetof(rlcs_call, %s));\n' % cname.get(f, f)
                              for f in fields)
                    + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I",
                    "/usr/local/cuda/include", str(prog), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == ct.sizeof(RlcsCall)
    assert got[1:] == [getattr(RlcsCall, f).offset for f in fields]


def _call(est, N=4, T=8, **ptrs):
    from linear_recurrence_scan_affine_gb300.binding import RlcsCall, GROUP_ESTIMATORS
    c = RlcsCall()
    c.estimator = GROUP_ESTIMATORS[est] if isinstance(est, str) else est
    for k, v in ptrs.items():
        setattr(c, k, v.value if isinstance(v, ctypes.c_void_p) else v)
    c.N, c.T, c.gamma, c.lambda_, c.rho_bar, c.c_bar = N, T, 0.99, 0.95, 1.0, 1.0
    return c


def _group(lib, calls, ws=None, wsb=0):
    from linear_recurrence_scan_affine_gb300.binding import RlcsCall
    arr = (RlcsCall * max(1, len(calls)))(*calls)
    return lib.rlcs_run_group(ctypes.cast(arr, ctypes.c_void_p), len(calls), ws, wsb, None)


def _group_ws(lib, calls):
    from linear_recurrence_scan_affine_gb300.binding import RlcsCall
    arr = (RlcsCall * max(1, len(calls)))(*calls)
    return lib.rlcs_group_workspace_bytes(ctypes.cast(arr, ctypes.c_void_p), len(calls))


def test_group_workspace_bytes(lib):
    assert _group_ws(lib, []) == 0
    a = [fake(i) for i in range(4)]
    gae = dict(rewards=a[0], values=a[1], terminateds=a[2], out=a[3])
    assert _group_ws(lib, [_call("gae", T=512, **gae)]) == 0       # short rows: none
    assert _group_ws(lib, [_call("gae", T=1000, **gae)]) == 0      # one tile per row: none
    # the tile length follows the group's rows: 4 rows alone take 4096-step
    # tiles, 4 + 1000 rows 2048-step ones
    one = _group_ws(lib, [_call("gae", N=4, T=16384, **gae)])
    assert one == 64 + 32 * 4 * 4
    two = _group_ws(lib, [_call("gae", N=4, T=16384, **gae),
                          _call("gae", N=1000, T=600, **gae)])
    assert two == 64 + 32 * 4 * 8


def test_group_validation(lib):
    # every case is rejected before anything is launched
    a = [fake(i) for i in range(12)]
    gae = dict(rewards=a[0], values=a[1], terminateds=a[2], out=a[3])
    assert lib.rlcs_run_group(None, 0, None, 0, None) == OK   # nothing to do
    assert lib.rlcs_run_group(None, 2, None, 0, None) == INVALID
    assert lib.rlcs_run_group(None, -1, None, 0, None) == INVALID
    assert _group(lib, [_call("gae", **gae)] * 17) == INVALID  # more than RLCS_MAX_GROUP
    # long rows that span several tiles need the group's workspace
    long = [_call("gae", T=50000, **gae)]
    assert _group_ws(lib, long) == 64 + 32 * 4 * 13  # 4096-step tiles: 13 per row
    assert _group(lib, long) == WORKSPACE
    assert _group(lib, long, fake(11, 1 << 30), _group_ws(lib, long) - 32) == WORKSPACE
    assert _group(lib, long, ctypes.c_void_p(a[0].value + 16), 1 << 20) == INVALID  # overlaps
    assert _group(lib, [_call(99, **gae)]) == INVALID           # unknown estimator
    bad = _call("gae", **gae)
    bad.reserved = 1
    assert _group(lib, [bad]) == INVALID
    # the namesake's own checks: a missing input, half a truncation pair, aliasing
    assert _group(lib, [_call("gae", rewards=a[0], terminateds=a[2], out=a[3])]) == INVALID
    assert _group(lib, [_call("gae", truncateds=a[4], **gae)]) == INVALID
    assert _group(lib, [_call("gae", rewards=a[0], values=a[1], terminateds=a[2],
                              out=a[1])]) == INVALID
    assert _group(lib, [_call("gae_and_returns", **gae)]) == INVALID  # returns missing
    # one call writing what another reads or writes (they run concurrently)
    other = dict(rewards=a[5], values=a[6], terminateds=a[7], out=a[8])
    assert _group(lib, [_call("gae", **gae),
                        _call("lambda_returns", **dict(other, out=a[0]))]) == INVALID
    assert _group(lib, [_call("gae", **gae),
                        _call("lambda_returns", **dict(other, out=a[3]))]) == INVALID
    inner = ctypes.c_void_p(a[2].value + 64)
    assert _group(lib, [_call("gae", **gae),
                        _call("discounted_returns", rewards=a[5], terminateds=a[7],
                              out=inner)]) == INVALID


def test_device_rollout_draws_the_named_fields():
    # the generator the size tests use on the GPU, exercised on the host
    import torch
    from synthetic_rollouts import device_rollout
    g = device_rollout(torch, 5, 7, 3, 0.3, ("rewards", "terminateds", "x_int", "bootstrap_value"),
                       "cpu")
    assert g["rewards"].shape == (5, 7) and g["rewards"].dtype == torch.float32
    assert g["x_int"].dtype == torch.int32 and int(g["x_int"].abs().max()) <= 100
    assert set(g["terminateds"].unique().tolist()) <= {0.0, 1.0}
    assert g["bootstrap_value"].shape == (5,)
    tm = device_rollout(torch, 5, 7, 3, 0.3, ("rewards",), "cpu", time_major=True)
    assert tm["rewards"].shape == (7, 5)
    again = device_rollout(torch, 5, 7, 3, 0.3, ("rewards",), "cpu")
    assert torch.equal(again["rewards"], g["rewards"])  # seeded
