"""The attention kernels' key-tile walk, compiled for the host, against the
oracle's tile_visits on many shapes (no GPU).

Every role of the attention kernels walks the ring with the same code
(csrc/ring_iter.cuh: segment ownership, segment and tile lengths clipped at
S, the ring order of steps and segments, causal skipping) on a geometry the
host planner (csrc/plan.cpp) builds. tests/iter_harness.cpp compiles both
unchanged with g++ and walks one query tile as a kernel does. The GPU visit
log checks the same walk on a few shapes; here it is compared entry by entry
-- (step, source rank, key tile id, FULL/PARTIAL) -- with oracle.tile_visits
for even and uneven lengths, every P up to 8, both orders, causal or not,
both tile heights, single ring steps, and packed sequences, including
malformed offset tables (which the kernels clamp). The backward's dK/dV
kernel walks the other way -- for one key tile, every query tile that sees
it, in the order the travelling block meets them (csrc/q_iter.cuh) -- and is
compared with the same oracle table read by key tile. The rows every load
and store addresses (seg_rows, lse_base) are checked against the three
layouts' definitions. The checked build's range checks (csrc/checks.cuh) are
built the same way: the tensor extents of each layout and the boundary of a
check.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle.schedule import segment_length

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sequence_exact_attention_gb300", "csrc")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
ORDERS = {"contiguous": 0, "zigzag": 1}
ORACLE_ORDER = {"contiguous": oracle.ORDER_CONTIGUOUS, "zigzag": oracle.ORDER_ZIGZAG}
CAP = 1 << 16


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are not available")
    out = str(tmp_path_factory.mktemp("iter") / "libiter.so")
    cmd = [gxx, "-std=c++17", "-O1", "-shared", "-fPIC", "-I", CSRC,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "iter_harness.cpp"), os.path.join(CSRC, "plan.cpp"),
           "-L", os.path.join(CUDA, "lib64"), "-Wl,-rpath," + os.path.join(CUDA, "lib64"),
           "-lcudart", "-o", out]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    lib = ctypes.CDLL(out)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.ra_test_geometry.argtypes = [ctypes.c_int] * 4 + [ip]
    lib.ra_test_walk.argtypes = [ctypes.c_int] * 7 + [ip, ctypes.c_int]
    lib.ra_test_block_walk.argtypes = [ctypes.c_int] * 6 + [ip, ctypes.c_int]
    lib.ra_test_walk_varlen.argtypes = ([ip] + [ctypes.c_int] * 10 + [ip, ctypes.c_int, ip, ip])
    lib.ra_test_extents.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_longlong)]
    lib.ra_test_qwalk.argtypes = [ctypes.c_int] * 6 + [ip, ctypes.c_int]
    lib.ra_test_varlen_status.argtypes = [ip] + [ctypes.c_int] * 4
    lp = ctypes.POINTER(ctypes.c_longlong)
    lib.ra_test_rows.argtypes = [ctypes.c_int] * 11 + [lp, lp, ctypes.c_int]
    lib.ra_test_in_range.argtypes = [ctypes.c_longlong] * 3 + [ip]
    return lib


def _buf(n):
    return (ctypes.c_int * n)()


def _walk(lib, S, P, causal, order, tile, step, qid):
    out = _buf(4 * CAP)
    n = lib.ra_test_walk(S, P, int(causal), ORDERS[order], tile, step, qid, out, CAP)
    assert 0 <= n <= CAP
    return [tuple(out[4 * i:4 * i + 4]) for i in range(n)]


def _geometry(lib, S, P, order, tile):
    f = _buf(3)
    assert lib.ra_test_geometry(S, P, ORDERS[order], tile, f) == 0
    return f[0], f[1], f[2]


def _check_all_tiles(lib, S, P, causal, order, tile, step=-1):
    want = oracle.tile_visits(S, P, causal, ORACLE_ORDER[order], tile)
    seg_len, n_seg, nt = _geometry(lib, S, P, order, tile)
    assert seg_len == segment_length(S, P, ORACLE_ORDER[order])
    assert len(want) == n_seg * nt
    for qid, w in enumerate(want):
        if step >= 0:
            w = [e for e in w if e[0] == step]
        got = _walk(lib, S, P, causal, order, tile, step, qid)
        assert got == [tuple(e) for e in w], (S, P, causal, order, tile, step, qid)


SMALL_S = [1, 2, 5, 63, 64, 65, 127, 128, 129, 255, 256, 300, 777, 1000, 1001, 1023]


@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_walk_matches_oracle_small(harness, order, causal, P):
    for S in SMALL_S:
        for tile in (64, 128):
            _check_all_tiles(harness, S, P, causal, order, tile)


@pytest.mark.parametrize("S,P,order", [(4096, 8, "contiguous"), (4100, 8, "zigzag"),
                                       (16384, 4, "contiguous"), (32760, 8, "zigzag"),
                                       (32768, 8, "zigzag")])
def test_walk_matches_oracle_workload_sizes(harness, S, P, order):
    _check_all_tiles(harness, S, P, True, order, 128)


@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
def test_single_step_walk_is_that_step_of_the_ring(harness, order):
    for S in (300, 1001):
        for P in (2, 4):
            for t in range(P):
                _check_all_tiles(harness, S, P, True, order, 128, step=t)
                _check_all_tiles(harness, S, P, False, order, 64, step=t)


def _check_blocks(lib, S, P, causal, order, step=-1):
    """The forward kernel pairs query tiles 2i and 2i+1 of a segment in one
    block walking the key tiles of the higher tile with tokens. Each tile's
    own walk (the oracle's tile visits) must be that block walk with the key
    tiles wholly after the tile left out, in the same order; the closed-form
    walk length the MMA issuers use must equal the walk's length."""
    tile = 128
    want = oracle.tile_visits(S, P, causal, ORACLE_ORDER[order], tile)
    seg_len, n_seg, nt = _geometry(lib, S, P, order, tile)
    for seg in range(n_seg):
        for ti in range(0, nt, 2):
            qid = seg * nt + ti
            out = _buf(4 * CAP)
            n = lib.ra_test_block_walk(S, P, int(causal), ORDERS[order], step, qid, out, CAP)
            assert 0 <= n <= CAP, (S, P, causal, order, step, qid, n)
            blk = [tuple(out[4 * i:4 * i + 4]) for i in range(n)]
            for k in (0, 1):
                if ti + k >= nt:
                    continue
                lo = seg * seg_len + (ti + k) * tile
                rows = min(tile, min(S, (seg + 1) * seg_len) - lo)
                w = [tuple(e[:3]) for e in want[qid + k] if step < 0 or e[0] == step]
                if rows <= 0:
                    assert w == []
                    continue
                hi = lo + rows - 1
                mine = [e[:3] for e in blk if not (causal and e[3] > hi)]
                assert mine == w, (S, P, causal, order, step, qid, k)


@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
def test_block_walk_covers_both_tiles(harness, order, causal):
    for S in (1, 5, 127, 128, 129, 255, 256, 257, 300, 600, 777, 1001, 4096, 4100):
        for P in (1, 2, 3, 4, 8):
            _check_blocks(harness, S, P, causal, order)
    for t in range(4):
        _check_blocks(harness, 1001, 4, causal, order, step=t)
    _check_blocks(harness, 32768, 8, causal, order)


def _clamped_length(cu, b, total, max_seqlen):
    lo = min(max(int(cu[b]), 0), total)
    hi = min(max(int(cu[b + 1]), lo), total)
    return lo, min(hi - lo, max_seqlen)


def _check_varlen(lib, cu, total, max_seqlen, P, causal, order, tile):
    n_seq = len(cu) - 1
    carr = (ctypes.c_int * len(cu))(*[int(x) for x in cu])
    # the grid's geometry: sized by max_seqlen
    _, n_seg, nt_grid = _geometry(lib, max_seqlen, P, order, tile)
    for b in range(n_seq):
        row0_want, S_b = _clamped_length(cu, b, total, max_seqlen)
        want = oracle.tile_visits(S_b, P, causal, ORACLE_ORDER[order], tile) if S_b > 0 else []
        seg_len_b = -(-S_b // n_seg)             # ceil: the sequence's own chunks
        nt_b = -(-seg_len_b // tile)
        for seg in range(n_seg):
            for ti in range(nt_grid):
                out, row0, facts = _buf(4 * CAP), ctypes.c_int(), _buf(3)
                n = lib.ra_test_walk_varlen(carr, n_seq, total, max_seqlen, P, int(causal),
                                            ORDERS[order], tile, b, seg, ti, out, CAP,
                                            ctypes.byref(row0), facts)
                assert row0.value == row0_want and facts[0] == S_b
                got = [tuple(out[4 * i:4 * i + 4]) for i in range(n)]
                if ti < nt_b:
                    assert got == [tuple(e) for e in want[seg * nt_b + ti]], (cu, b, seg, ti)
                else:
                    assert got == [], (cu, b, seg, ti)      # a tile past the sequence


@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_walk_is_each_sequences_own_ring(harness, order, causal):
    lengths = [300, 0, 1, 777, 128, 1000]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    _check_varlen(harness, cu, int(cu[-1]), max(lengths), 4, causal, order, 128)
    _check_varlen(harness, cu, int(cu[-1]), max(lengths), 3, causal, order, 64)


@pytest.mark.parametrize("cu,total,max_seqlen", [
    ([0, 500, 300, 900], 900, 600),     # decreasing offset: an empty sequence
    ([0, 400, 1200], 1000, 800),        # past the tensors' end: clipped at total
    ([-50, 200, 260], 260, 300),        # negative offset: clamped to 0
    ([0, 700, 900], 900, 256),          # longer than max_seqlen: clipped to it
])
def test_varlen_walk_clamps_malformed_tables(harness, cu, total, max_seqlen):
    _check_varlen(harness, np.asarray(cu), total, max_seqlen, 2, True, "zigzag", 128)


@pytest.mark.parametrize("layout", [0, 1, 2])
def test_checked_build_extents(harness, layout):
    B, H_q, H_kv, S, D, P, total = 3, 8, 2, 1001, 128, 4, 2500
    ext = (ctypes.c_longlong * 3)()
    assert harness.ra_test_extents(layout, B, H_q, H_kv, S, D, P, total, ext) == 0
    # rows of the call's layout: B*S, the packed total, or P shards of ceil(S/P) per batch
    rows = {0: B * S, 1: total, 2: P * B * (-(-S // P))}[layout]
    assert list(ext) == [rows * H_q * D, rows * H_kv * D, rows * H_q]


def test_checked_build_range_boundary(harness):
    st = ctypes.c_int(0)
    assert harness.ra_test_in_range(0, 10, 10, ctypes.byref(st)) == 1
    assert harness.ra_test_in_range(9, 1, 10, ctypes.byref(st)) == 1
    assert st.value == 0
    assert harness.ra_test_in_range(9, 2, 10, ctypes.byref(st)) == 0
    assert st.value == 10                     # RA_ERR_RANGE
    st.value = 0
    assert harness.ra_test_in_range(-1, 1, 10, ctypes.byref(st)) == 0
    assert st.value == 10
    assert harness.ra_test_in_range(5, 1, 10, None) == 1
    assert harness.ra_test_in_range(50, 1, 10, None) == 0     # no status word: only skipped


def _qwalk_expected(S, P, causal, order, tile):
    """For every key tile, the (step, query segment, query tile, masked)
    entries of the query tiles that visit it, from oracle.tile_visits,
    ordered by ring step and then by query position."""
    visits = oracle.tile_visits(S, P, causal, ORACLE_ORDER[order], tile)
    nt = -(-segment_length(S, P, ORACLE_ORDER[order]) // tile)
    by_key = {}
    for qid, vs in enumerate(visits):
        for t, _src, kid, cls in vs:
            by_key.setdefault(kid, []).append((t, qid // nt, qid % nt,
                                               int(cls == oracle.PARTIAL)))
    return {kid: sorted(e) for kid, e in by_key.items()}, len(visits)


@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_backward_walk_matches_oracle(harness, order, causal, P):
    for S in SMALL_S + [4100]:
        for tile in (64, 128):
            want, n_tiles = _qwalk_expected(S, P, causal, order, tile)
            for kid in range(n_tiles):
                out = _buf(4 * CAP)
                n = harness.ra_test_qwalk(S, P, int(causal), ORDERS[order], tile, kid, out, CAP)
                got = [tuple(out[4 * i:4 * i + 4]) for i in range(n)]
                assert got == want.get(kid, []), (S, P, causal, order, tile, kid)


def _rows(lib, layout, B, H_q, S, P, order, total, row0, b, h, seg):
    n_max = S + 1
    rows, lse = (ctypes.c_longlong * n_max)(), (ctypes.c_longlong * n_max)()
    n = lib.ra_test_rows(layout, B, H_q, S, P, ORDERS[order], total, row0, b, h, seg, rows,
                         lse, n_max)
    assert n >= 0
    return list(rows[:n]), list(lse[:n])


@pytest.mark.parametrize("S,P", [(1000, 4), (1001, 4), (256, 2), (5, 4), (4100, 8)])
def test_row_addressing_of_every_layout(harness, S, P):
    """The rows the kernels load and store, in each layout, restated from the
    layouts' definitions: [B, S, H, D] with lse [B, H, S]; packed rows from
    the sequence's first row with lse [H, total]; the sequence-parallel
    [P, B, C, H, D] (C = ceil(S/P), shard p = positions pC ..) with lse
    [P, B, H, C]."""
    B, H = 3, 2
    for order in ("contiguous", "zigzag"):
        parts = 2 * P if order == "zigzag" else P
        seg_len = -(-S // parts)
        for seg in range(parts):
            positions = list(range(seg * seg_len, min(S, (seg + 1) * seg_len)))
            for b in range(B):
                for h in range(H):
                    got = _rows(harness, 0, B, H, S, P, order, 0, 0, b, h, seg)
                    assert got == ([b * S + p for p in positions],
                                   [(b * H + h) * S + p for p in positions])
                    total, row0 = 5000, 17 + 100 * b
                    got = _rows(harness, 1, B, H, S, P, order, total, row0, b, h, seg)
                    assert got == ([row0 + p for p in positions],
                                   [h * total + row0 + p for p in positions])
        # the sharded layout exists for contiguous chunks only (shard p = chunk p)
        C = -(-S // P)
        for p in range(P):
            positions = list(range(p * C, min(S, (p + 1) * C)))
            for b in range(B):
                for h in range(H):
                    got = _rows(harness, 2, B, H, S, P, "contiguous", 0, 0, b, h, p)
                    assert got == ([(p * B + b) * C + (x - p * C) for x in positions],
                                   [((p * B + b) * H + h) * C + (x - p * C)
                                    for x in positions])


@pytest.mark.parametrize("cu,total,max_seqlen,b,flagged", [
    ((0, 100, 300), 300, 200, 0, False),       # well formed
    ((0, 100, 300), 300, 200, 1, False),
    ((0, 100, 350), 300, 250, 1, True),        # last offset past total
    ((0, 250, 300), 300, 200, 0, True),        # a sequence longer than max_seqlen
    ((0, 120, 100, 300), 300, 200, 1, True),   # decreasing offsets
    ((-5, 100, 300), 300, 200, 0, True),       # negative first offset
])
def test_checked_build_reports_clamped_offsets(harness, cu, total, max_seqlen, b, flagged):
    """The checked build sets RA_ERR_RANGE when the packed offsets need
    clamping (the release build clamps silently), so a caller can tell a
    malformed cu_seqlens from a good run."""
    carr = (ctypes.c_int * len(cu))(*cu)
    st = harness.ra_test_varlen_status(carr, len(cu) - 1, total, max_seqlen, b)
    assert st == (10 if flagged else 0)
