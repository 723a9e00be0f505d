// schedule.h -- the tile schedule of the grouped-GEMM kernels as pure
// functions, compiled both into the kernels (device) and into host code (the
// scheduler's enumeration test builds this header with a plain C++ compiler).
//
// What is scheduled (SkyRL PR #867, "Integrate ragged_dot pallas kernel with
// group_offset support": the suggested fast_ragged_dot body -- group
// boundaries from a cumulative sum with an initial zero, only the local groups
// [group_offset, group_offset + g_local) computed, the other rows zeroed;
// MaxText PR #5760, "MoE wo FSDP sharding and valid-rows-only MoE kernels":
// rows [0, limit) only):
//   * group boundaries bound[i] = min(sum_{j<i} max(size_j, 0), L);
//   * forward / dx: ceil(rows_j / TM) x n_tiles output tiles per local group,
//     visited in bands of band_tiles m-tiles (inside a band the m-tiles run
//     fastest and the band sweeps every column tile); the last m-tile of a
//     group is loaded from end - TM, so no loaded row reaches the group end;
//   * dw: dw_m_tiles x n_tiles tiles per local group; the contraction runs
//     over the group's rows in 64-row K blocks, the last one loaded from
//     end - 64 with the rows before the group skipped (whole 16-row steps) or
//     zeroed (the straddling step);
//   * zero fill (forward / dx): rows [0, zero_lo) and [zero_hi, L) split into
//     contiguous 16-byte shares, one per CTA.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define RD_HD __host__ __device__ __forceinline__
#else
#define RD_HD inline
#endif

namespace rd {

enum GemmOp : int {
  kOpFwd = 0,  // out[i] = lhs[i] @ rhs[j]             (A K-major, B MN-major)
  kOpDx = 1,   // out[i] = lhs[i] @ rhs[j]^T           (A K-major, B K-major)
  kOpDw = 2    // out[j] = x[rows_j]^T @ y[rows_j]     (A MN-major, B MN-major)
};

constexpr int kBM = 128;   // accumulator rows per CTA
constexpr int kBN = 256;   // accumulator columns
constexpr int kBK = 64;    // K block (one 128-byte swizzle atom of bf16)

// One unit of work as every role of the kernel sees it.
struct Tile {
  int32_t j;         // local group
  int32_t m_idx;     // row tile (fwd/dx: within the group; dw: within the weight block)
  int32_t n_idx;     // column tile
  int32_t rs, re;    // rows of the group, clamped to L
  int32_t row_load;  // fwd/dx: first row the tile's A rows are loaded from
  int32_t nkb;       // K blocks (0: the tile is all zeros)
};

// The schedule's inputs: the boundary and tile-prefix arrays plus the sizes.
struct SchedView {
  const int32_t* bound;       // [g_total + 1] group boundaries, clamped to L
  const int32_t* tile_start;  // fwd/dx: [g_local + 1] first tile of each local group;
                              // dw: [g_local] the local group at each position of the
                              // tile order (groups without rows first)
  int32_t group_offset;
  int32_t g_local;
  int32_t n_tiles;
  int32_t band_tiles;   // fwd/dx
  int32_t dw_m_tiles;   // dw
  int32_t kc;           // fwd/dx contraction length
};

// dw visits the groups without rows first: their tiles only write zeros (no
// MMA), so handing them out at the start lets those writes overlap the first
// real tiles and leaves the real tiles evenly spread over the CTAs.
RD_HD bool group_is_empty(const int32_t* bound, int group_offset, int j) {
  return bound[group_offset + j + 1] == bound[group_offset + j];
}

RD_HD int32_t clamp_boundary(long long run, int32_t L) {
  return static_cast<int32_t>(run < L ? run : L);
}

// Tiles of local group j whose rows are [lo, hi).
RD_HD long long tiles_of_group(int op, int32_t lo, int32_t hi, int tm, int32_t n_tiles,
                               int32_t dw_m_tiles) {
  if (op == kOpDw) return static_cast<long long>(dw_m_tiles) * n_tiles;
  const int32_t cnt = hi - lo;
  return static_cast<long long>((cnt + tm - 1) / tm) * n_tiles;
}

template <int OP, int TM>
RD_HD Tile decode_tile_view(const SchedView& v, int t) {
  Tile tl;
  if (OP == kOpDw) {
    const int per_group = v.dw_m_tiles * v.n_tiles;
    const int pos = t / per_group;
    tl.j = v.tile_start[pos];
    const int u = t - pos * per_group;
    tl.m_idx = u % v.dw_m_tiles;
    tl.n_idx = u / v.dw_m_tiles;
    tl.rs = v.bound[v.group_offset + tl.j];
    tl.re = v.bound[v.group_offset + tl.j + 1];
    tl.row_load = 0;
    tl.nkb = (tl.re - tl.rs + kBK - 1) / kBK;
  } else {
    int lo = 0, hi = v.g_local;  // tile_start[lo] <= t < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (v.tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    tl.j = lo;
    const int u = t - v.tile_start[lo];
    tl.rs = v.bound[v.group_offset + lo];
    tl.re = v.bound[v.group_offset + lo + 1];
    // Bands of band_tiles m-tiles: within a band the m-tiles run fastest and the
    // band sweeps every n-tile before the next band starts, so the band's lhs
    // rows stay in L2 while each rhs column panel is read once per band.
    const int kBand = v.band_tiles;
    const int mt = (tl.re - tl.rs + TM - 1) / TM;
    const int band = u / (kBand * v.n_tiles);
    const int rem = u - band * kBand * v.n_tiles;
    const int left = mt - band * kBand;
    const int bw = kBand < left ? kBand : left;
    tl.m_idx = band * kBand + rem % bw;
    tl.n_idx = rem / bw;
    const int first = tl.rs + tl.m_idx * TM;
    tl.row_load = (tl.m_idx == mt - 1) ? tl.re - TM : first;
    tl.nkb = (v.kc + kBK - 1) / kBK;
  }
  return tl;
}

// forward / dx: the rows a tile stores are [store_lo, store_hi); its A rows
// are loaded from [row_load, row_load + TM).
RD_HD int32_t tile_store_lo(const Tile& tl, int tm) { return tl.rs + tl.m_idx * tm; }
RD_HD int32_t tile_store_hi(const Tile& tl) { return tl.re; }

// dw: first row of K block kb of a tile (the last block is loaded from end - 64).
RD_HD int32_t dw_block_row(const Tile& tl, int kb) {
  return (kb == tl.nkb - 1) ? tl.re - kBK : tl.rs + kb * kBK;
}

// dw: rows of the last K block of a group that precede the block's own start
// (the block is loaded from row end - 64).  Whole 16-row K steps of them are
// skipped by the MMA; the rows of the step that straddles the start must be
// zeroed in shared memory.  Returns the first K step to issue and sets
// [z0, z1) to the rows to zero (empty when z0 == z1).
RD_HD int dw_edge(const Tile& tl, int kb, int& z0, int& z1) {
  z0 = z1 = 0;
  if (kb != tl.nkb - 1) return 0;
  const int rem = (tl.re - tl.rs) - (tl.nkb - 1) * kBK;
  const int zrows = kBK - rem;
  z0 = zrows & ~15;
  z1 = zrows;
  return zrows >> 4;
}

// dw through per-group tensor maps (the map's rows are the group's rows, so
// rows outside the group are out of bounds and land as zeros): the K blocks
// are aligned to end at the group end, block kb starting at group row
// rem - 64 + 64 kb with rem = the rows of the last block (1..64); the first
// block's rows above the group start arrive as zeros, and its whole 16-row
// steps of them are skipped.  Returns the first K step to issue; *row
// receives the block's first row relative to the group start.
RD_HD int dw_group_block(const Tile& tl, int kb, int* row) {
  const int rem = (tl.re - tl.rs) - (tl.nkb - 1) * kBK;
  *row = rem - kBK + kb * kBK;
  return kb == 0 ? (kBK - rem) >> 4 : 0;
}

// Zero fill: the 16-byte units [u0, u1) of the zero rows that one CTA writes.
// Units (CTAs or CTA pairs) with one tile fewer than the others (u >= r, r =
// total % units) take twice the share: they have a tile's time to spare at
// the end.  In a pair each CTA takes half of its unit's share.
RD_HD void zero_share(uint64_t units16, int unit, int units, int total_tiles, bool pair,
                      int sub, uint64_t& u0, uint64_t& u1) {
  const int r = total_tiles % units;
  auto W = [&](int u) -> uint64_t {
    return (r == 0 || u <= r) ? static_cast<uint64_t>(u)
                              : static_cast<uint64_t>(r + 2 * (u - r));
  };
  const uint64_t wt = W(units);
  const uint64_t a0 = units16 * W(unit) / wt, a1 = units16 * W(unit + 1) / wt;
  const uint64_t per_unit = pair ? 2 : 1, s = pair ? static_cast<uint64_t>(sub) : 0;
  u0 = a0 + (a1 - a0) * s / per_unit;
  u1 = a0 + (a1 - a0) * (s + 1) / per_unit;
}

}  // namespace rd
