"""Host-side checks of the C ABI (no GPU needed).

  * the library loads and exports every function include/muon_ns.h declares;
  * argument validation returns the documented status codes before touching a
    device;
  * the tile scheduler (the kernels' own decode, through the ABI) covers every
    output tile of a launch exactly once, and a model of the epilogue's store
    predicates writes every output element exactly once, in bounds.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import newton_schulz_07_gb300 as ns
from newton_schulz_07_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon_ns.h")
TILE_M, TILE_N = 128, 256


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    L = _lib.lib()
    declared = header_functions()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(L, name), f"{name} declared in muon_ns.h but not exported"
    assert set(declared) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_version_and_status_strings():
    L = _lib.lib()
    assert L.muon_ns_version().decode() == ns.__version__
    for code in range(7):
        assert L.muon_ns_status_string(code)
    assert L.muon_ns_status_string(99).decode() == "unknown status"


def test_launch_count():
    L = _lib.lib()
    assert [L.muon_ns_launches_per_call(s) for s in (0, 1, 5)] == [2, 4, 16]
    assert L.muon_ns_launches_per_call(-1) == -1


def _ws(b, r, c):
    n = ctypes.c_size_t(0)
    s = _lib.lib().muon_ns_workspace_size(b, r, c, ctypes.byref(n))
    return s, n.value


def test_workspace_size_and_regions():
    s, total = _ws(4, 256, 512)
    assert s == _lib.OK
    regions = {}
    for reg in range(7):
        regions[reg] = ns.workspace_region(4, 256, 512, reg)
    assert regions[_lib.WS_TOTAL] == (0, total)
    assert regions[_lib.WS_X][1] == 4 * 256 * 512 * 2
    assert regions[_lib.WS_GRAM][1] == regions[_lib.WS_POLY][1] == 4 * 256 * 256 * 2
    assert regions[_lib.WS_DIAG][1] == 4 * 256 * 4
    # Regions are disjoint, aligned and inside the workspace.
    spans = sorted((o, o + n) for r, (o, n) in regions.items() if r != _lib.WS_TOTAL)
    for (o0, e0), (o1, _) in zip(spans, spans[1:]):
        assert e0 <= o1
    for r in (_lib.WS_X, _lib.WS_GRAM, _lib.WS_POLY):
        assert regions[r][0] % 1024 == 0
        assert regions[r][0] + regions[r][1] <= total
    # Tall input: the Gram is cols x cols.
    assert ns.workspace_region(2, 512, 256, _lib.WS_GRAM)[1] == 2 * 256 * 256 * 2
    assert _ws(0, 256, 512) == (_lib.OK, 0)


@pytest.mark.parametrize("b,r,c,code", [
    (-1, 8, 8, _lib.ERR_INVALID_ARG),
    (1, -8, 8, _lib.ERR_INVALID_ARG),
    (1, 12, 16, _lib.ERR_ALIGNMENT),
    (1, 16, 20, _lib.ERR_ALIGNMENT),
    (1, (1 << 20) + 8, 8, _lib.ERR_INVALID_ARG),
    (1, 65536, 65536, _lib.ERR_INVALID_ARG),
])
def test_shape_validation(b, r, c, code):
    assert _ws(b, r, c)[0] == code
    L = _lib.lib()
    p = ctypes.c_void_p(4096)
    assert L.muon_ns_ws(p, p, b, r, c, 5, None, 1e-7, p, 1 << 40, None) == code
    assert L.muon_ns(p, p, b, r, c, 5, None, 1e-7, None) == code


def _call_ws(**kw):
    L = _lib.lib()
    args = dict(G=4096, out=4096, batch=2, rows=64, cols=128, steps=5, coeffs=None, eps=1e-7,
                ws=4096, wsb=1 << 30, stream=None)
    args.update(kw)
    cf = None
    if args["coeffs"] is not None:
        cf = ctypes.cast((ctypes.c_float * 3)(*args["coeffs"]), ctypes.POINTER(ctypes.c_float))
    return L.muon_ns_ws(ctypes.c_void_p(args["G"]), ctypes.c_void_p(args["out"]), args["batch"], args["rows"],
                        args["cols"], args["steps"], cf, args["eps"], ctypes.c_void_p(args["ws"]),
                        args["wsb"], args["stream"])


def test_argument_validation_codes():
    assert _call_ws(G=0) == _lib.ERR_INVALID_ARG
    assert _call_ws(out=0) == _lib.ERR_INVALID_ARG
    assert _call_ws(steps=-1) == _lib.ERR_INVALID_ARG
    assert _call_ws(eps=-1.0) == _lib.ERR_INVALID_ARG
    assert _call_ws(eps=float("nan")) == _lib.ERR_INVALID_ARG
    assert _call_ws(eps=float("inf")) == _lib.ERR_INVALID_ARG
    assert _call_ws(coeffs=(1.0, float("nan"), 1.0)) == _lib.ERR_INVALID_ARG
    assert _call_ws(G=4098) == _lib.ERR_ALIGNMENT
    assert _call_ws(out=4104) == _lib.ERR_ALIGNMENT
    assert _call_ws(ws=0) == _lib.ERR_WORKSPACE
    assert _call_ws(wsb=16) == _lib.ERR_WORKSPACE
    assert _call_ws(ws=4096 + 16) == _lib.ERR_ALIGNMENT
    # Empty problems succeed without touching pointers or the device.
    assert _call_ws(G=0, out=0, ws=0, batch=0) == _lib.OK
    assert _call_ws(G=0, out=0, ws=0, rows=0) == _lib.OK
    L = _lib.lib()
    assert L.muon_ns_gram(None, None, 1, 16, 12, None, 0.0, None, None) == _lib.ERR_ALIGNMENT
    assert L.muon_ns_gram(None, None, 1, 16, 16, None, 0.0, None, None) == _lib.ERR_INVALID_ARG
    p8 = ctypes.c_void_p(8192)
    assert L.muon_ns_gram(ctypes.c_void_p(4096), p8, 1, 16, 16, p8, -1.0, None, None) == _lib.ERR_INVALID_ARG
    p = ctypes.c_void_p(4096)
    assert L.muon_ns_poly(p, p, None, 1, 16, 1.0, 1.0, None, None) == _lib.ERR_INVALID_ARG  # B == A
    assert L.muon_ns_poly(p, ctypes.c_void_p(8192), ctypes.c_void_p(12), 1, 16, 1.0, 1.0, None,
                          None) == _lib.ERR_ALIGNMENT  # diag not 16-byte aligned
    assert L.muon_ns_update(p, ctypes.c_void_p(8192), None, p, 1, 16, 16, 1.0, None, 0.0, None,
                            None) == _lib.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_is_unsupported():
    assert _call_ws() == _lib.ERR_UNSUPPORTED_DEVICE
    assert _lib.lib().muon_ns_device_supported(-1) == _lib.ERR_UNSUPPORTED_DEVICE


# ---------------------------------------------------------------- scheduler --

def tiles(kind, batch, M, N):
    L = _lib.lib()
    total = L.muon_ns_tile_count(kind, batch, M, N)
    b, i, j = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    out = []
    for t in range(total):
        assert L.muon_ns_tile_coords(kind, batch, M, N, t, ctypes.byref(b), ctypes.byref(i), ctypes.byref(j)) == 0
        out.append((b.value, i.value, j.value))
    return out


SYM_SIZES = [8, 120, 128, 136, 248, 256, 264, 384, 392, 512, 640, 768, 1000, 1536, 2056]


@pytest.mark.parametrize("m", SYM_SIZES)
def test_triangle_schedule_covers_lower_triangle_once(m):
    ts = tiles(0, 2, m, m)
    tm = -(-m // TILE_M)
    T = -(-m // TILE_N)
    expect = {(b, I, J) for b in range(2) for I in range(tm) for J in range(T) if J <= I // 2}
    assert len(ts) == len(set(ts)) == len(expect)
    assert set(ts) == expect
    # Matrix-major order.
    assert [b for b, _, _ in ts] == sorted(b for b, _, _ in ts)


def test_triangle_tile_counts():
    L = _lib.lib()
    assert L.muon_ns_tile_count(0, 128, 1536, 1536) == 128 * 42
    assert L.muon_ns_tile_count(0, 1, 8192, 8192) == 32 * 33
    assert L.muon_ns_tile_count(0, 1, 768, 768) == 12
    assert L.muon_ns_tile_count(0, 1, 16, 8) == -1


@pytest.mark.parametrize("M,N", [(8, 8), (128, 256), (136, 264), (1536, 2048), (2048, 768), (400, 1000),
                                 (1100, 520)])
def test_grid_schedule_covers_every_tile_once(M, N):
    ts = tiles(1, 3, M, N)
    tm, tn = -(-M // TILE_M), -(-N // TILE_N)
    expect = {(b, I, J) for b in range(3) for I in range(tm) for J in range(tn)}
    assert len(ts) == len(set(ts)) and set(ts) == expect


def unpair(units, M):
    """Row tiles the two CTAs of a cluster compute for paired units (b, p, J):
    2p and 2p + 1, the latter only if it exists (otherwise nothing is stored)."""
    tm = -(-M // TILE_M)
    return [(b, 2 * p + r, J) for b, p, J in units for r in (0, 1) if 2 * p + r < tm]


@pytest.mark.parametrize("m", SYM_SIZES)
def test_paired_triangle_schedule_covers_lower_triangle_once(m):
    ts = unpair(tiles(2, 2, m, m), m)
    tm = -(-m // TILE_M)
    T = -(-m // TILE_N)
    expect = {(b, I, J) for b in range(2) for I in range(tm) for J in range(T) if J <= I // 2}
    assert len(ts) == len(set(ts)) == len(expect)
    assert set(ts) == expect
    assert [b for b, _, _ in ts] == sorted(b for b, _, _ in ts)


@pytest.mark.parametrize("M,N", [(8, 8), (128, 256), (136, 264), (1536, 2048), (2048, 768), (400, 1000),
                                 (1100, 520), (7168, 2048)])
def test_paired_grid_schedule_covers_every_tile_once(M, N):
    ts = unpair(tiles(3, 3, M, N), M)
    tm, tn = -(-M // TILE_M), -(-N // TILE_N)
    expect = {(b, I, J) for b in range(3) for I in range(tm) for J in range(tn)}
    assert len(ts) == len(set(ts)) and set(ts) == expect


@pytest.mark.parametrize("kind,M,N", [(2, 1536, 1536), (2, 1000, 1000), (2, 8, 8), (3, 1536, 2048),
                                      (3, 2048, 768), (3, 1096, 1304), (3, 136, 264)])
def test_paired_units_per_matrix_match_single_matrix_count(kind, M, N):
    # A whole call's per-matrix completion counters expect, after each step of
    # a product, the single-matrix unit count of its tile space (times a fixed
    # increment per unit): every matrix of a stack must own exactly that many.
    batch = 3
    per = _lib.lib().muon_ns_tile_count(kind, 1, M, N)
    counts = np.bincount([b for b, _, _ in tiles(kind, batch, M, N)], minlength=batch)
    assert per > 0 and list(counts) == [per] * batch


def test_paired_tile_counts():
    L = _lib.lib()
    assert L.muon_ns_tile_count(2, 128, 1536, 1536) == 128 * 21  # 6 pair rows: 6 * 7 / 2
    assert L.muon_ns_tile_count(2, 1, 8192, 8192) == 32 * 33 // 2
    assert L.muon_ns_tile_count(3, 128, 1536, 2048) == 128 * 6 * 8
    assert L.muon_ns_tile_count(3, 1, 136, 264) == 1 * 2  # one pair row (row tiles 0, 1), two column tiles
    assert L.muon_ns_tile_count(2, 1, 16, 8) == -1
    assert L.muon_ns_tile_count(4, 1, 16, 16) == -1


def _epilogue_writes(kind, M, N, ts):
    """Model of the epilogue store predicates: counts how often each output
    element is written (direct and mirrored stores) over all tiles."""
    count = np.zeros((M, N), dtype=np.int32)
    r = np.arange(TILE_M)[:, None]
    c = np.arange(TILE_N)[None, :]
    for _, I, J in ts:
        gi = I * TILE_M + r
        gj = J * TILE_N + c
        inb = (gi < M) & (gj < N)
        if kind == 1:
            np.add.at(count, (np.broadcast_to(gi, inb.shape)[inb], np.broadcast_to(gj, inb.shape)[inb]), 1)
            continue
        d = inb & (gj <= gi)
        np.add.at(count, (np.broadcast_to(gi, d.shape)[d], np.broadcast_to(gj, d.shape)[d]), 1)
        mi = inb & (gj < gi)
        np.add.at(count, (np.broadcast_to(gj, mi.shape)[mi], np.broadcast_to(gi, mi.shape)[mi]), 1)
    return count


@pytest.mark.parametrize("m", [8, 136, 256, 392, 640, 1000])
def test_symmetric_epilogue_writes_each_element_once(m):
    ts = [t for t in tiles(0, 1, m, m)]
    assert np.all(_epilogue_writes(0, m, m, ts) == 1)
    assert np.all(_epilogue_writes(0, m, m, unpair(tiles(2, 1, m, m), m)) == 1)


@pytest.mark.parametrize("M,N", [(8, 8), (136, 264), (400, 1000)])
def test_full_epilogue_writes_each_element_once(M, N):
    assert np.all(_epilogue_writes(1, M, N, tiles(1, 1, M, N)) == 1)


def _chunk_store_writes(m, ts, warps_per_quarter=2):
    """Model of the symmetric epilogue's bulk stores: per 32-row warp block and
    32-column chunk, the chunk (below the diagonal) plus its transpose, or the
    symmetrised diagonal block; counts writes per 32 x 32 block."""
    nb = -(-m // 32)
    count = np.zeros((nb, nb), dtype=np.int32)
    for _, I, J in ts:
        for q in range(4):
            R0 = I * TILE_M + q * 32
            if R0 >= m:
                continue  # all rows clipped
            for cc in range(TILE_N // 32):
                gj0 = J * TILE_N + cc * 32
                if gj0 >= m or gj0 > R0 + 31:
                    break
                if gj0 < R0:
                    count[R0 // 32, gj0 // 32] += 1
                    count[gj0 // 32, R0 // 32] += 1
                else:
                    count[R0 // 32, R0 // 32] += 1
    return count


@pytest.mark.parametrize("m", [8, 136, 256, 392, 640, 1000, 1536])
def test_symmetric_bulk_stores_write_each_block_once(m):
    assert np.all(_chunk_store_writes(m, tiles(0, 1, m, m)) == 1)


def test_grouped_workspace_is_sum_of_stack_workspaces():
    shapes = [(3, 136, 264), (2, 264, 136), (0, 8, 8), (1, 392, 392)]
    arr = (_lib.MuonNSStack * len(shapes))()
    for i, (b, r, c) in enumerate(shapes):
        arr[i] = _lib.MuonNSStack(4096, 4096, b, r, c)
    n = ctypes.c_size_t(0)
    L = _lib.lib()
    assert L.muon_ns_grouped_workspace_size(arr, len(shapes), ctypes.byref(n)) == _lib.OK
    assert n.value == sum(_ws(b, r, c)[1] for b, r, c in shapes)
    arr[1] = _lib.MuonNSStack(4096, 4096, 2, 264, 130)
    assert L.muon_ns_grouped_workspace_size(arr, len(shapes), ctypes.byref(n)) == _lib.ERR_ALIGNMENT
    assert L.muon_ns_grouped(arr, 65, 5, None, 1e-7, ctypes.c_void_p(4096), 1 << 30, None) == _lib.ERR_INVALID_ARG
    assert L.muon_ns_grouped(None, 0, 5, None, 1e-7, None, 0, None) == _lib.OK
    arr[1] = _lib.MuonNSStack(4096, 0, 2, 264, 136)
    assert L.muon_ns_grouped(arr, len(shapes), 5, None, 1e-7, ctypes.c_void_p(4096), 1 << 30,
                             None) == _lib.ERR_INVALID_ARG
    arr[1] = _lib.MuonNSStack(4096, 4096, 2, 264, 136)
    assert L.muon_ns_grouped(arr, len(shapes), 5, None, 1e-7, ctypes.c_void_p(4096), 16, None) == _lib.ERR_WORKSPACE


def test_f32_workspace_regions_hold_fp32():
    n = ctypes.c_size_t(0)
    assert _lib.lib().muon_ns_f32_workspace_size(4, 256, 512, ctypes.byref(n)) == _lib.OK
    assert ns.f32_workspace_region(4, 256, 512, _lib.WS_X)[1] == 4 * 256 * 512 * 4
    assert ns.f32_workspace_region(4, 256, 512, _lib.WS_GRAM)[1] == 4 * 256 * 256 * 4
    assert ns.f32_workspace_region(4, 256, 512, _lib.WS_TOTAL)[1] == n.value > _ws(4, 256, 512)[1]
    L = _lib.lib()
    p = ctypes.c_void_p(4096)
    assert L.muon_ns_ws_f32(p, p, 1, 12, 16, 5, None, 1e-7, p, 1 << 30, None) == _lib.ERR_ALIGNMENT
    assert L.muon_ns_ws_f32(p, p, 1, 16, 16, 5, None, 1e-7, p, 16, None) == _lib.ERR_WORKSPACE


# ---------------------------------------------------------- host-held stacks --

def _call_host(**kw):
    L = _lib.lib()
    args = dict(G=4096, out=4096, batch=16, rows=64, cols=128, steps=5, eps=1e-7, chunk=0,
                ws=4096, wsb=1 << 30, stream=None)
    args.update(kw)
    return L.muon_ns_host(ctypes.c_void_p(args["G"]), ctypes.c_void_p(args["out"]), args["batch"], args["rows"],
                          args["cols"], args["steps"], None, args["eps"], args["chunk"], ctypes.c_void_p(args["ws"]),
                          args["wsb"], args["stream"])


def test_host_path_workspace_arithmetic():
    def ws(b, r, c, chunk=0):
        return ns.host_workspace_size(b, r, c, chunk)
    one = ns.workspace_size(1, 256, 512)
    # error word + 2 slots of (input chunk, output chunk, NS workspace of a chunk)
    for chunk in (1, 3, 16):
        slot = 2 * chunk * 256 * 512 * 2 + ns.workspace_size(chunk, 256, 512)
        assert 2 * slot <= ws(16, 256, 512, chunk) <= 2 * slot + 1024 + 4 * 1024
    # Default largest chunk: the whole stack under 32 MiB ...
    assert ws(16, 256, 512) == ws(16, 256, 512, 16)
    # ... else about 96 MiB of input (16 matrices of 1536 x 2048, 4 of 7168 x 2048) ...
    assert ws(128, 1536, 2048) == ws(128, 1536, 2048, 16)
    assert ws(32, 7168, 2048) == ws(32, 7168, 2048, 4)
    # ... but at most half the stack.
    assert ws(16, 1536, 2048) == ws(16, 1536, 2048, 8)
    assert ws(17, 1536, 2048) == ws(17, 1536, 2048, 9)
    assert [ns.host_chunk(*s) for s in [(16, 256, 512), (128, 1536, 2048), (32, 7168, 2048),
                                        (128, 2048, 768), (16, 1536, 2048), (1, 8192, 8192)]] == [16, 16, 4, 32, 8, 1]
    assert ns.host_chunk(128, 1536, 2048, 5) == 5 and ns.host_chunk(4, 256, 512, 100) == 4
    assert ns.host_chunk(0, 256, 512) == 0 and ns.host_chunk(2, 12, 8) == 0
    assert ws(4, 256, 512, 100) == ws(4, 256, 512, 4)   # clamped to the batch
    assert ws(16, 256, 512, 4) > ws(16, 256, 512, 2) > one
    assert ws(0, 256, 512) == 0


def test_host_plan_covers_the_stack():
    # Explicit chunk: half-size ends around full chunks, the remainder before the last.
    assert ns.host_plan(10, 136, 264, 3) == [2, 3, 3, 2]
    assert ns.host_plan(10, 136, 264, 4) == [2, 4, 2, 2]
    assert ns.host_plan(10, 136, 264, 9) == [5, 5]
    assert ns.host_plan(10, 136, 264, 100) == [10]
    # Default largest chunk, same shape of plan.
    assert ns.host_plan(128, 1536, 2048) == [8] + [16] * 7 + [8]
    assert ns.host_plan(32, 7168, 2048) == [2] + [4] * 7 + [2]
    assert ns.host_plan(128, 2048, 768) == [16, 32, 32, 32, 16]
    assert ns.host_plan(16, 1536, 2048) == [4, 8, 4]
    assert ns.host_plan(16, 256, 512) == [16]  # under 32 MiB: one chunk
    for shape in [(128, 1536, 2048), (32, 7168, 2048), (128, 2048, 768), (16, 1536, 2048), (17, 1536, 2048),
                  (3, 4096, 4096), (1, 8192, 8192), (1000, 1024, 1024), (10, 136, 264)]:
        for chunk in (0, 1, 2, 3, 7, 16):
            plan = ns.host_plan(*shape, chunk)
            c = ns.host_chunk(*shape, chunk)
            assert sum(plan) == shape[0] and all(1 <= v <= c for v in plan), (shape, chunk, plan)
            assert len(plan) == 1 or plan[0] == plan[-1] == (c + 1) // 2
    assert ns.host_plan(0, 256, 512) == []
    with pytest.raises(ValueError):
        ns.host_plan(2, 12, 8)


def test_host_path_argument_errors():
    assert _call_host(G=0) == _lib.ERR_INVALID_ARG
    assert _call_host(out=0) == _lib.ERR_INVALID_ARG
    assert _call_host(rows=60) == _lib.ERR_ALIGNMENT
    assert _call_host(steps=-1) == _lib.ERR_INVALID_ARG
    assert _call_host(batch=-1) == _lib.ERR_INVALID_ARG
    assert _call_host(wsb=1024) == _lib.ERR_WORKSPACE
    assert _call_host(ws=0) == _lib.ERR_WORKSPACE
    assert _call_host(ws=4096 + 16) == _lib.ERR_ALIGNMENT
    assert _call_host(batch=0) == _lib.OK  # empty stack: nothing to do


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_host_path_without_device_is_unsupported():
    assert _call_host() == _lib.ERR_UNSUPPORTED_DEVICE


def test_wait_budget_and_stall_injection_settings():
    # Host-side settings only: no device needed.
    L = _lib.lib()
    assert L.muon_ns_set_wait_budget(-1) == _lib.ERR_INVALID_ARG
    assert L.muon_ns_set_wait_budget(20_000_000) == _lib.OK
    assert L.muon_ns_set_wait_budget(0) == _lib.OK
    assert L.muon_ns_inject_stall(1) == _lib.OK
    assert L.muon_ns_inject_stall(0) == _lib.OK


# ----------------------------------------------------------------- Muon step --

def _call_step(**kw):
    # Fake, distinct, 16-byte aligned addresses: every check below returns
    # before the library touches a device or dereferences a pointer.
    L = _lib.lib()
    args = dict(W=1 << 20, M=2 << 20, G=3 << 20, batch=2, rows=64, cols=128, steps=5, eps=1e-7,
                ws=1 << 24, wsb=1 << 30, hp=_lib.MuonStepHparams(0.02, 0.95, 0.0, 1.0, 1))
    args.update(kw)
    hp = args["hp"]
    return L.muon_step_ws(ctypes.c_void_p(args["W"]), ctypes.c_void_p(args["M"]), ctypes.c_void_p(args["G"]),
                          args["batch"], args["rows"], args["cols"], None if hp is None else ctypes.byref(hp),
                          args["steps"], None, ctypes.c_float(args["eps"]), ctypes.c_void_p(args["ws"]), args["wsb"],
                          None)


def test_muon_step_argument_errors():
    nan = float("nan")
    assert _call_step(W=0) == _lib.ERR_INVALID_ARG
    assert _call_step(M=0) == _lib.ERR_INVALID_ARG
    assert _call_step(G=0) == _lib.ERR_INVALID_ARG
    assert _call_step(hp=None) == _lib.ERR_INVALID_ARG
    for bad in (_lib.MuonStepHparams(nan, 0.95, 0.0, 1.0, 1), _lib.MuonStepHparams(0.02, float("inf"), 0.0, 1.0, 1),
                _lib.MuonStepHparams(0.02, 0.95, nan, 1.0, 1), _lib.MuonStepHparams(0.02, 0.95, 0.0, nan, 1)):
        assert _call_step(hp=bad) == _lib.ERR_INVALID_ARG
    nbytes = 4 * 2 * 64 * 128
    assert _call_step(M=(1 << 20) + nbytes - 16) == _lib.ERR_INVALID_ARG  # W and M overlap
    assert _call_step(G=(2 << 20) + 16) == _lib.ERR_INVALID_ARG  # M and G overlap
    assert _call_step(W=(1 << 20) + 4) == _lib.ERR_ALIGNMENT
    assert _call_step(rows=60) == _lib.ERR_ALIGNMENT
    assert _call_step(steps=-1) == _lib.ERR_INVALID_ARG
    assert _call_step(eps=-1.0) == _lib.ERR_INVALID_ARG
    assert _call_step(wsb=1024) == _lib.ERR_WORKSPACE
    assert _call_step(ws=0) == _lib.ERR_WORKSPACE
    assert _call_step(ws=(1 << 24) + 16) == _lib.ERR_ALIGNMENT
    assert _call_step(batch=0) == _lib.OK  # empty stack: nothing to do


def test_muon_step_workspace_and_launch_count():
    ws = ns.step_workspace_size(2, 64, 128)
    # The NS workspace of the stack, then U (bf16) rounded up to 1 KiB.
    assert ws == -(-ns.workspace_size(2, 64, 128) // 1024) * 1024 + -(-(2 * 2 * 64 * 128) // 1024) * 1024
    assert ns.step_workspace_size(0, 64, 128) == 0
    assert ns.step_launches(5) == 16 and ns.step_launches(0) == 3 and ns.step_launches(-1) == -1
    assert ns.default_scale(2048, 768) == (2048 / 768) ** 0.5 and ns.default_scale(768, 2048) == 1.0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_muon_step_without_device_is_unsupported():
    assert _call_step() == _lib.ERR_UNSUPPORTED_DEVICE


def test_header_compiles_as_c_and_cpp(tmp_path):
    # The boundary is a C ABI: the header must stand alone in a C99 and a C++17
    # translation unit that uses its types and entry points.
    import shutil
    import subprocess

    cuda_inc = "/usr/local/cuda/include"
    cc, cxx = shutil.which("gcc"), shutil.which("g++")
    if not (cc and cxx and os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h"))):
        pytest.skip("no host C compiler or CUDA headers")
    src = tmp_path / "use_header.c"
    src.write_text('#include "muon_ns.h"\n'
                   "int main(void) {\n"
                   "  muon_step_hparams h = {0.02f, 0.95f, 0.0f, 1.0f, 1};\n"
                   "  muon_ns_stack s = {0, 0, 1, 8, 8};\n"
                   "  size_t n = 0;\n"
                   "  (void)h; (void)s;\n"
                   "  return muon_ns_workspace_size(1, 8, 8, &n) + muon_step_workspace_size(1, 8, 8, &n);\n"
                   "}\n")
    inc = ["-I" + os.path.join(ROOT, "include"), "-I" + cuda_inc]
    for cmd in ([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only"] + inc + [str(src)],
                [cxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++"] + inc + [str(src)]):
        p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        assert p.returncode == 0, p.stdout


def _step_stack_array(specs):
    arr = (_lib.MuonStepStack * max(len(specs), 1))()
    for i, (W, M, G, b, r, c) in enumerate(specs):
        arr[i] = _lib.MuonStepStack(W, M, G, b, r, c, _lib.MuonStepHparams(0.02, 0.95, 0.0, 1.0, 1))
    return arr


def test_grouped_step_workspace_and_errors():
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    MB = 1 << 20
    specs = [(1 * MB, 2 * MB, 3 * MB, 2, 64, 128), (4 * MB, 5 * MB, 6 * MB, 3, 136, 264), (0, 0, 0, 0, 64, 128)]
    arr = _step_stack_array(specs)
    assert L.muon_step_grouped_workspace_size(arr, 3, ctypes.byref(n)) == _lib.OK
    assert n.value == ns.step_workspace_size(2, 64, 128) + ns.step_workspace_size(3, 136, 264)

    def call(specs, wsb=1 << 30, ws=1 << 24):
        a = _step_stack_array(specs)
        return L.muon_step_grouped(a, len(specs), 5, None, ctypes.c_float(1e-7), ctypes.c_void_p(ws), wsb, None)

    # The second stack's W overlaps the first stack's G (read while it is written).
    assert call([specs[0], (3 * MB + 64, 5 * MB, 6 * MB, 3, 136, 264)]) == _lib.ERR_INVALID_ARG
    # W and M of one stack overlap.
    assert call([(1 * MB, 1 * MB + 16, 3 * MB, 2, 64, 128)]) == _lib.ERR_INVALID_ARG
    assert call([(0, 2 * MB, 3 * MB, 2, 64, 128)]) == _lib.ERR_INVALID_ARG
    assert call([(1 * MB + 4, 2 * MB, 3 * MB, 2, 64, 128)]) == _lib.ERR_ALIGNMENT
    assert call([(1 * MB, 2 * MB, 3 * MB, 2, 60, 128)]) == _lib.ERR_ALIGNMENT
    assert call(specs[:2], wsb=1024) == _lib.ERR_WORKSPACE
    assert call(specs[:2], ws=(1 << 24) + 16) == _lib.ERR_ALIGNMENT
    assert call([specs[2]]) == _lib.OK  # only an empty stack: nothing to do
    assert L.muon_step_grouped(None, 1, 5, None, ctypes.c_float(1e-7), None, 0, None) == _lib.ERR_INVALID_ARG
    big = (_lib.MuonStepStack * 65)()
    assert L.muon_step_grouped(big, 65, 5, None, ctypes.c_float(1e-7), None, 0, None) == _lib.ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert call(specs[:2]) == _lib.ERR_UNSUPPORTED_DEVICE


def _half_store_writes(m, ts, sm2):
    """Model of the symmetric epilogue's bulk stores with half storage: per
    32-row warp block and 32-column chunk, the chunk alone outside the
    diagonal 256-blocks; inside them, on 2-SM units (which compute the whole
    block), every chunk as computed, and otherwise the chunk below the
    diagonal plus its transpose, or the symmetrised diagonal block.  Counts
    writes per 32 x 32 block."""
    nb = -(-m // 32)
    count = np.zeros((nb, nb), dtype=np.int32)
    for _, I, J in ts:
        for q in range(4):
            R0 = I * TILE_M + q * 32
            if R0 >= m:
                continue  # all rows clipped
            direct = sm2 and (J * TILE_N) >> 8 == R0 >> 8
            for cc in range(TILE_N // 32):
                gj0 = J * TILE_N + cc * 32
                if gj0 >= m or (gj0 > R0 + 31 and not direct):
                    break
                if direct or (gj0 < R0 and gj0 >> 8 != R0 >> 8):
                    count[R0 // 32, gj0 // 32] += 1
                elif gj0 < R0:
                    count[R0 // 32, gj0 // 32] += 1
                    count[gj0 // 32, R0 // 32] += 1
                else:
                    count[R0 // 32, R0 // 32] += 1
    return count


@pytest.mark.parametrize("m", [8, 136, 256, 392, 640, 1000, 1040, 1536])
@pytest.mark.parametrize("sm2", [False, True])
def test_half_storage_writes_lower_triangle_and_diagonal_blocks_once(m, sm2):
    # Half storage must hold every 32 x 32 block of the lower triangle and of
    # the diagonal 256-blocks exactly once, and nothing else, whether the
    # units are 2-SM pairs (direct stores inside the diagonal blocks) or
    # single / multicast tiles (mirrored stores there).
    nb = -(-m // 32)
    bi, bj = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    want = ((bj <= bi) | ((bi * 32) >> 8 == (bj * 32) >> 8)).astype(np.int32)
    units = unpair(tiles(2, 1, m, m), m)
    np.testing.assert_array_equal(_half_store_writes(m, units, sm2), want)
    if not sm2:
        np.testing.assert_array_equal(_half_store_writes(m, tiles(0, 1, m, m), False), want)


def test_half_storage_flags():
    # Unknown flag bits are refused before the device is queried; the half
    # flag itself is valid (without a GPU the call then stops at the device).
    L = _lib.lib()
    p = 1 << 20
    assert L.muon_ns_gram_ex(p, p, 1, 256, 512, None, 1e-7, 2, None, None) == _lib.ERR_INVALID_ARG
    assert L.muon_ns_poly_ex(p, p + 4096, None, 1, 256, -4.775, 2.0315, 4, None, None) == _lib.ERR_INVALID_ARG
    assert L.muon_ns_update_ex(p, p + 4096, None, p + 8192, 1, 256, 512, 3.4445, None, 1e-7, 3, None,
                               None) == _lib.ERR_INVALID_ARG
    assert L.muon_ns_gram_ex(p, p, 1, 256, 512, None, 1e-7, _lib.HALF, None, None) == _lib.ERR_UNSUPPORTED_DEVICE
