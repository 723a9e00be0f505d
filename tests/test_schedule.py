"""The grouped-GEMM tile schedule, enumerated on the host.

The kernels take their tile arithmetic from ``csrc/schedule.h`` (pure
``__host__ __device__`` functions).  ``sched_probe.cpp`` compiles that header
with the host C++ compiler; this test enumerates every tile of a launch for
many random size vectors (empty groups, negative and overflowing sizes,
offsets, limits, bands of one to many tiles, both tile heights) and checks
what the kernels rely on:

* the boundaries equal the oracle's (cumulative sum with an initial zero,
  clamped to L);
* forward / dx: every (group, m-tile, n-tile) appears exactly once; for each
  column tile the rows the tiles store partition the group's rows exactly; no
  tile loads a row at or past its group's end (hence none at or past L);
* dw: every (m-tile, n-tile) of every local group appears exactly once, and
  the rows its K blocks feed to the MMA (after skipping and zeroing the rows
  before the group in the last block) are the group's rows, each once; no
  block loads a row at or past the group's end;
* zero fill: the CTAs' shares partition the zero rows exactly.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "expert_ffn_ragged_gb300", "csrc")
OP_FWD, OP_DX, OP_DW = 0, 1, 2


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    out = str(tmp_path_factory.mktemp("sched") / "libsched_probe.so")
    src = os.path.join(ROOT, "tests", "sched_probe.cpp")
    subprocess.run([cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-I" + CSRC, src, "-o", out],
                   check=True)
    lib = ctypes.CDLL(out)
    lib.sched_tiles.restype = ctypes.c_longlong
    lib.sched_tiles.argtypes = [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 10 + \
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong]
    lib.sched_dw_block.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p]
    lib.sched_zero_share.argtypes = [ctypes.c_ulonglong] + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    lib.sched_dw_group_block.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


def _tiles(lib, op, sizes, m, limit, off, gl, tm, n_tiles, band_tiles=1, dw_m_tiles=0, kc=64):
    sizes = np.ascontiguousarray(sizes, dtype=np.int32)
    g = sizes.size
    bound = np.zeros(g + 1, np.int32)
    cap = 1 << 20
    tiles = np.zeros((cap, 9), np.int32)
    n = lib.sched_tiles(op, sizes.ctypes.data, g, m, -1 if limit is None else limit, off, gl, tm,
                        n_tiles, band_tiles, dw_m_tiles, kc, bound.ctypes.data, tiles.ctypes.data,
                        cap)
    assert n >= 0
    return bound, tiles[:n]


def _random_case(rng):
    g = int(rng.integers(1, 40))
    sizes = rng.integers(0, 1500, g)
    sizes[rng.random(g) < 0.25] = 0                      # empty groups
    if rng.random() < 0.2:
        sizes[rng.integers(0, g)] = -int(rng.integers(1, 50))   # a negative size
    total = int(np.maximum(sizes, 0).sum())
    m = max(1, total + int(rng.integers(-200, 300)))     # sometimes the sizes overflow m
    limit = None if rng.random() < 0.4 else int(rng.integers(0, m + 50))
    off = int(rng.integers(0, g))
    gl = int(rng.integers(1, g - off + 1))
    return sizes.astype(np.int32), m, limit, off, gl


@pytest.mark.parametrize("op", [OP_FWD, OP_DX])
@pytest.mark.parametrize("tm", [128, 256])
def test_forward_tiles_cover_each_output_block_once(probe, op, tm):
    rng = np.random.default_rng(100 + op * 7 + tm)
    for case in range(150):
        sizes, m, limit, off, gl = _random_case(rng)
        n_tiles = int(rng.integers(1, 6))
        band = int(rng.choice([1, 2, 3, 5, 16, 1 << 20]))
        bound, tiles = _tiles(probe, op, sizes, m, limit, off, gl, tm, n_tiles, band_tiles=band)
        b, L = oracle.group_bounds(sizes, m, limit)
        np.testing.assert_array_equal(bound, b)
        expect = sum(-(-(int(b[off + j + 1]) - int(b[off + j])) // tm) * n_tiles for j in range(gl))
        assert len(tiles) == expect, case
        keys = set()
        cover = {}
        for (j, mi, ni, rs, re, row_load, nkb, lo, hi) in tiles.tolist():
            assert 0 <= j < gl and 0 <= ni < n_tiles
            assert (rs, re) == (b[off + j], b[off + j + 1])
            mt = -(-(re - rs) // tm)
            assert 0 <= mi < mt
            assert (j, mi, ni) not in keys
            keys.add((j, mi, ni))
            assert row_load + tm <= re, "a tile loads a row at or past its group's end"
            assert re <= L
            s0, s1 = max(lo, row_load), min(hi, row_load + tm)
            assert s1 > s0
            cover.setdefault((j, ni), []).append((s0, s1))
        for (j, ni), spans in cover.items():
            spans.sort()
            assert spans[0][0] == b[off + j] and spans[-1][1] == b[off + j + 1]
            for (a0, a1), (c0, c1) in zip(spans, spans[1:]):
                assert a1 == c0, f"rows stored twice or never in group {j} column tile {ni}"


def test_band_order_visits_m_tiles_fastest(probe):
    """Inside a band the m-tiles run fastest; the band sweeps every column tile first."""
    sizes = np.array([1500, 700], np.int32)
    _, tiles = _tiles(probe, OP_FWD, sizes, 2200, None, 0, 2, 128, 3, band_tiles=4)
    g0 = tiles[tiles[:, 0] == 0]
    order = [(int(mi), int(ni)) for mi, ni in g0[:, 1:3]]
    # 12 m-tiles in bands 4, 4, 4 over 3 column tiles
    want = [(band * 4 + r, ni) for band in range(3) for ni in range(3) for r in range(4)]
    assert order == want


@pytest.mark.parametrize("tm", [128, 256])
def test_dw_blocks_feed_each_group_row_once(probe, tm):
    rng = np.random.default_rng(7 + tm)
    blk = np.zeros(4, np.int32)
    for case in range(80):
        sizes, m, limit, off, gl = _random_case(rng)
        n_tiles, dw_m_tiles = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        bound, tiles = _tiles(probe, OP_DW, sizes, m, limit, off, gl, tm, n_tiles,
                              dw_m_tiles=dw_m_tiles)
        b, L = oracle.group_bounds(sizes, m, limit)
        np.testing.assert_array_equal(bound, b)
        assert len(tiles) == gl * n_tiles * dw_m_tiles
        keys = {(int(j), int(mi), int(ni)) for j, mi, ni in tiles[:, :3]}
        assert keys == {(j, mi, ni) for j in range(gl) for mi in range(dw_m_tiles)
                        for ni in range(n_tiles)}
        # groups without rows come first in the tile order, each part in index order
        seq = [int(j) for j in tiles[::n_tiles * dw_m_tiles, 0]]
        empty = [j for j in range(gl) if b[off + j + 1] == b[off + j]]
        assert seq == empty + [j for j in range(gl) if j not in empty]
        checked = set()
        for (j, _, _, rs, re, _, nkb, _, _) in tiles.tolist():
            if j in checked:
                continue
            checked.add(j)
            assert nkb == -(-(re - rs) // 64)
            fed = []
            for kb in range(nkb):
                probe.sched_dw_block(rs, re, kb, blk.ctypes.data)
                row0, kk0, z0, z1 = (int(x) for x in blk)
                assert row0 + 64 <= re, "a K block loads a row at or past the group's end"
                assert z0 == 16 * kk0 and z0 <= z1 <= 63
                # steps before kk0 are not issued; rows [z0, z1) are zeroed
                fed += list(range(row0 + z1, row0 + 64))
            assert sorted(fed) == list(range(rs, re)), f"group {j}: rows fed to the MMA"


def test_dw_group_map_blocks(probe):
    """dw through per-group maps: the blocks end at the group end; rows above the group
    start (negative, out of the map's bounds, zero-filled) lie only in the first block;
    after the skipped whole steps every group row is fed once and no row past it."""
    out = np.zeros(2, np.int32)
    for cnt in list(range(1, 300)) + [1023, 1024, 1025, 1170, 4096]:
        nkb = -(-cnt // 64)
        fed = []
        for kb in range(nkb):
            probe.sched_dw_group_block(cnt, kb, out.ctypes.data)
            row, kk0 = int(out[0]), int(out[1])
            assert row + 64 <= cnt, "a block reads past the group"
            if kb > 0:
                assert row >= 0 and kk0 == 0
            else:
                assert -64 < row <= 0 and row + 16 * kk0 > -16 and row + 16 * kk0 <= 0
            fed += [r for r in range(row + 16 * kk0, row + 64) if r >= 0]
        assert fed == list(range(cnt))


def test_zero_fill_shares_partition_the_zero_rows(probe):
    rng = np.random.default_rng(3)
    out = np.zeros(2, np.uint64)
    for _ in range(300):
        units16 = int(rng.integers(0, 1 << 24))
        units = int(rng.integers(1, 153))
        total = int(rng.integers(0, 5000))
        pair = bool(rng.integers(0, 2))
        pos = 0
        for u in range(units):
            for sub in (range(2) if pair else range(1)):
                probe.sched_zero_share(units16, u, units, total, int(pair), sub, out.ctypes.data)
                u0, u1 = int(out[0]), int(out[1])
                assert u0 == pos and u1 >= u0
                pos = u1
        assert pos == units16
