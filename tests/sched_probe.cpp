// sched_probe.cpp -- host build of the grouped-GEMM tile schedule for the
// enumeration test (tests/test_schedule.py).  It compiles the kernels' own
// schedule header (expert_ffn_ragged_gb300/csrc/schedule.h) with a plain C++
// compiler and exposes it through a few C functions; the boundaries are
// built here sequentially, with the header's per-element formulas, where the
// kernel runs a warp scan.
#include <stdint.h>

#include "schedule.h"

using namespace rd;

namespace {

// boundaries clamped to L and the per-group tile prefix; returns the tile count
long long build(int op, const int32_t* sizes, int g_total, int m, int limit, int off, int gl,
                int tm, int n_tiles, int dw_m_tiles, int32_t* bound, int32_t* tile_start) {
  int32_t L = m;
  if (limit >= 0) L = limit > m ? m : limit;
  long long run = 0;
  for (int i = 0; i < g_total; ++i) {
    bound[i] = clamp_boundary(run, L);
    run += sizes[i] > 0 ? sizes[i] : 0;
  }
  bound[g_total] = clamp_boundary(run, L);
  long long t = 0;
  if (op == kOpDw) {
    // the group order of the dw tiles: groups without rows first
    int p = 0;
    for (int j = 0; j < gl; ++j)
      if (group_is_empty(bound, off, j)) tile_start[p++] = j;
    for (int j = 0; j < gl; ++j)
      if (!group_is_empty(bound, off, j)) tile_start[p++] = j;
    for (int j = 0; j < gl; ++j) t += tiles_of_group(op, 0, 0, tm, n_tiles, dw_m_tiles);
    return t;
  }
  for (int j = 0; j < gl; ++j) {
    tile_start[j] = static_cast<int32_t>(t);
    t += tiles_of_group(op, bound[off + j], bound[off + j + 1], tm, n_tiles, dw_m_tiles);
  }
  tile_start[gl] = static_cast<int32_t>(t);
  return t;
}

template <int OP, int TM>
void decode_all(const SchedView& v, long long total, int32_t* out) {
  for (long long t = 0; t < total; ++t) {
    const Tile tl = decode_tile_view<OP, TM>(v, static_cast<int>(t));
    int32_t* o = out + 9 * t;
    o[0] = tl.j;
    o[1] = tl.m_idx;
    o[2] = tl.n_idx;
    o[3] = tl.rs;
    o[4] = tl.re;
    o[5] = tl.row_load;
    o[6] = tl.nkb;
    o[7] = OP == kOpDw ? 0 : tile_store_lo(tl, TM);
    o[8] = OP == kOpDw ? 0 : tile_store_hi(tl);
  }
}

}  // namespace

extern "C" {

// Every tile of one launch, in tile-index order: 9 int32 per tile (j, m_idx,
// n_idx, rs, re, row_load, nkb, store_lo, store_hi).  bound receives the
// g_total + 1 boundaries.  Returns the tile count, or -1 if it exceeds cap.
long long sched_tiles(int op, const int32_t* sizes, int g_total, int m, int limit, int off, int gl,
                      int tm, int n_tiles, int band_tiles, int dw_m_tiles, int kc, int32_t* bound,
                      int32_t* tiles, long long cap) {
  static int32_t tile_start[1025];
  const long long total =
      build(op, sizes, g_total, m, limit, off, gl, tm, n_tiles, dw_m_tiles, bound, tile_start);
  if (total > cap) return -1;
  SchedView v;
  v.bound = bound;
  v.tile_start = tile_start;
  v.group_offset = off;
  v.g_local = gl;
  v.n_tiles = n_tiles;
  v.band_tiles = band_tiles;
  v.dw_m_tiles = dw_m_tiles;
  v.kc = kc;
  if (op == kOpDw) {
    if (tm == 256) decode_all<kOpDw, 256>(v, total, tiles);
    else decode_all<kOpDw, 128>(v, total, tiles);
  } else if (op == kOpDx) {
    if (tm == 256) decode_all<kOpDx, 256>(v, total, tiles);
    else decode_all<kOpDx, 128>(v, total, tiles);
  } else {
    if (tm == 256) decode_all<kOpFwd, 256>(v, total, tiles);
    else decode_all<kOpFwd, 128>(v, total, tiles);
  }
  return total;
}

// dw K block kb of a tile with rows [rs, re): out = (first loaded row, first
// 16-row step issued, z0, z1) with [z0, z1) the in-block rows zeroed.
void sched_dw_block(int rs, int re, int kb, int32_t* out) {
  Tile tl{};
  tl.rs = rs;
  tl.re = re;
  tl.nkb = (re - rs + kBK - 1) / kBK;
  int z0, z1;
  const int kk0 = dw_edge(tl, kb, z0, z1);
  out[0] = dw_block_row(tl, kb);
  out[1] = kk0;
  out[2] = z0;
  out[3] = z1;
}

// dw through per-group maps, block kb of a group of `cnt` rows: out = (first
// row relative to the group, first 16-row step issued).
void sched_dw_group_block(int cnt, int kb, int32_t* out) {
  Tile tl{};
  tl.rs = 0;
  tl.re = cnt;
  tl.nkb = (cnt + kBK - 1) / kBK;
  int row;
  out[1] = dw_group_block(tl, kb, &row);
  out[0] = row;
}

// The zero-fill share [u0, u1) of one CTA (unit, and sub = the CTA in a pair).
void sched_zero_share(unsigned long long units16, int unit, int units, int total_tiles, int pair,
                      int sub, unsigned long long* out) {
  uint64_t u0, u1;
  zero_share(units16, unit, units, total_tiles, pair != 0, sub, u0, u1);
  out[0] = u0;
  out[1] = u1;
}

}  // extern "C"
