// gemm_kernel.cuh -- the persistent tcgen05 grouped-GEMM kernel behind
// rd_ragged_dot (forward, optional fused SiLU-GLU), rd_ragged_dot_trans_rhs
// (dx) and rd_trans_ragged_dot (dw).
//
// What it computes (SkyRL PR #867, "Integrate ragged_dot pallas kernel with
// group_offset support": suggested fast_ragged_dot body and the
// trans_ragged_dot backward fix; MaxText PR #5760, "MoE wo FSDP sharding and
// valid-rows-only MoE kernels": commit message on rows [0, limit)):
//   forward  out[i]  = lhs[i] @ rhs[j]          for rows i of local group j
//   dx       out[i]  = lhs[i] @ rhs[j]^T
//   dw       out[j]  = x[rows_j]^T @ y[rows_j]
//   rows in [0, L) outside the local groups are +0, rows >= L untouched.
//
// How (persistent, 384 threads per CTA):
//   * every CTA reads group_sizes and *limit itself and builds the group
//     boundaries (exclusive prefix clamped to L) and the per-group tile
//     prefix in shared memory -- no workspace, no host round trip;
//   * tiles are handed out by static striding over (group, band, n-tile,
//     m-tile): within a band of rows (6144 by default) the m-tiles run
//     fastest, so the CTAs working at one time share each rhs column panel
//     through L2 and the band's lhs rows stay in L2 until every column panel
//     has used them;
//   * warp 0 (one lane) streams A/B blocks with TMA into a ring of
//     128-byte-swizzled tiles; one lane of warp 1 waits for each block,
//     issues its tcgen05.mma into one of two TMEM accumulators and commits;
//     warps 2-9 (two per TMEM lane quarter) drain the other accumulator with
//     tcgen05.ld, round to bf16 (or apply the GLU) and store full 64-byte row
//     segments through a small shared-memory transpose, with row masks;
//     warp 10 has the bulk-copy engine write the zero rows of the forward/dx
//     outputs from a zero block in shared memory, paced by the producer;
//   * PAIR=false: one CTA per SM computes a 128x256 tile (UMMA 128x256x16,
//     4-stage ring of 48 KB).  PAIR=true: a cluster of two CTAs computes a
//     256x256 tile with the CTA-pair UMMA (cta_group::2, 256x256x16): each
//     CTA loads its own 128 rows of A and its own 128 columns of B (32 KB per
//     stage, 6 stages), both CTAs' copies are counted on the even CTA's
//     barrier, the even CTA issues the MMA, and each CTA drains its own half
//     of the accumulator.  Half the B bytes per SM and more stages in flight;
//   * the last m-tile of a group is loaded from row (end - tile rows) so no
//     row at or past the group end -- hence none at or past L -- is read; it
//     stores only the rows it owns.  dw uses the same shift on its row (K)
//     blocks, skips whole 16-row K steps before the group and has warp 10
//     zero, in shared memory, the rows of the straddling step (NaN-safe);
//   * every wait is bounded; on expiry the CTA unwinds, drains its TMA and
//     MMA work, frees TMEM and reports RD_STATUS_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/rd.h"
#include "gemm_args.h"
#include "glu_math.cuh"
#include "ptx.cuh"

namespace rd {

// Bounds of the waits made while unwinding after a timeout: every copy or MMA
// still in flight then completes within microseconds.
constexpr uint64_t kDrainNs = 1000000000ull;
constexpr uint64_t kGraceNs = 200000ull;

template <bool PAIR>
struct TileCfg {
  static constexpr int kStagesN = PAIR ? 6 : 4;
  static constexpr int kTileM = PAIR ? 2 * kBM : kBM;   // rows of one (pair) tile
  static constexpr int kBCols = PAIR ? kBN / 2 : kBN;   // B columns held by one CTA
  static constexpr int kStageA = kBM * kBK * 2;         // 16 KB
  static constexpr int kStageB = kBCols * kBK * 2;      // 16 KB (pair) or 32 KB
  static constexpr int kStageBytes = kStageA + kStageB;
};

template <bool PAIR>
struct alignas(128) GemmShared {
  static constexpr int S = TileCfg<PAIR>::kStagesN;
  uint8_t mapstage[2][128];  // dw with group maps: the two maps being rebased (128-byte aligned)
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t efull[S];   // dw: this CTA's copy of an edge block landed (edge fills only)
  uint64_t pready[S];  // dw: the edge rows of this stage are zeroed (in a pair: in both CTAs)
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t L;
  int32_t total_tiles;
  int32_t zero_lo;  // forward/dx: rows [0, zero_lo) are zero
  int32_t zero_hi;  // forward/dx: rows [zero_hi, L) are zero
  int32_t fills;      // stages the producer has filled so far (paces the zero fill)
  int32_t maps_built;  // dw with group maps: tiles with rows whose maps are published
  int32_t bound[kMaxGroups + 1];       // group boundaries, clamped to L
  int32_t tile_start[kMaxGroups + 1];  // fwd/dx: first tile of each local group; dw: group order
  uint4 epi[kEpiWarps][32 * 4];        // epilogue staging per warp: 32 rows x 64 bytes
  uint4 zeros[256];                    // 4 KB zero block, the source of the zero-fill copies
};

template <bool PAIR>
constexpr size_t gemm_smem_bytes_t() {
  return 1024 + static_cast<size_t>(TileCfg<PAIR>::kStagesN) * TileCfg<PAIR>::kStageBytes +
         sizeof(GemmShared<PAIR>);
}

// Exclusive prefix of a per-lane chunk sum across one warp.
__device__ __forceinline__ long long warp_exclusive_scan(long long v, int lane) {
  long long incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  return incl - v;
}

// Run by one warp: group boundaries, tile prefix, zero ranges, status bits.
template <int OP, bool PAIR>
__device__ __forceinline__ void build_schedule(GemmShared<PAIR>& sh, const GemmArgs& a, int lane) {
  constexpr int TM = TileCfg<PAIR>::kTileM;
  int32_t L = a.m;
  if (a.limit != nullptr) {
    const int32_t v = *a.limit;
    L = v < 0 ? 0 : (v > a.m ? a.m : v);
  }
  // exclusive prefix of max(size, 0) over all g_total groups, clamped to L
  const int G = a.g_total;
  const int per = (G + 31) / 32;
  const int lo = min(lane * per, G), hi = min(lo + per, G);
  long long sum = 0;
  int neg = 0;
  for (int i = lo; i < hi; ++i) {
    const int s = a.group_sizes[i];
    neg |= s < 0;
    sum += s > 0 ? s : 0;
  }
  long long run = warp_exclusive_scan(sum, lane);
  for (int i = lo; i < hi; ++i) {
    sh.bound[i] = clamp_boundary(run, L);
    const int s = a.group_sizes[i];
    run += s > 0 ? s : 0;
  }
  const long long total = __shfl_sync(0xFFFFFFFFu, run, 31);
  neg = __any_sync(0xFFFFFFFFu, neg);
  if (lane == 0) {
    sh.bound[G] = clamp_boundary(total, L);
    sh.L = L;
    if (a.status != nullptr && blockIdx.x == 0) {
      int bits = 0;
      if (neg) bits |= RD_STATUS_NEG_SIZE;
      if (total > a.m) bits |= RD_STATUS_OVERFLOW;
      if (bits) atomicOr(a.status, bits);
    }
  }
  __syncwarp();
  // tiles of each local group
  const int GL = a.g_local;
  const int per2 = (GL + 31) / 32;
  const int lo2 = min(lane * per2, GL), hi2 = min(lo2 + per2, GL);
  auto tiles_of = [&](int j) -> long long {
    return tiles_of_group(OP, sh.bound[a.group_offset + j], sh.bound[a.group_offset + j + 1], TM,
                          a.n_tiles, a.dw_m_tiles);
  };
  if (OP == kOpDw) {
    // the tile order's group sequence: groups without rows first, each part in
    // index order (a warp partition: empties before this lane's chunk, and after)
    int n_empty = 0;
    for (int j = lo2; j < hi2; ++j) n_empty += group_is_empty(sh.bound, a.group_offset, j) ? 1 : 0;
    const int e_before = static_cast<int>(warp_exclusive_scan(n_empty, lane));
    const int e_total = __shfl_sync(0xFFFFFFFFu, e_before + n_empty, 31);
    int pe = e_before, pn = e_total + (lo2 - e_before);
    for (int j = lo2; j < hi2; ++j) {
      if (group_is_empty(sh.bound, a.group_offset, j)) sh.tile_start[pe++] = j;
      else sh.tile_start[pn++] = j;
    }
  }
  long long tsum = 0;
  for (int j = lo2; j < hi2; ++j) tsum += tiles_of(j);
  long long trun = warp_exclusive_scan(tsum, lane);
  if (OP != kOpDw) {
    for (int j = lo2; j < hi2; ++j) {
      sh.tile_start[j] = static_cast<int32_t>(trun);
      trun += tiles_of(j);
    }
  } else {
    trun += tsum;
  }
  const long long ttotal = __shfl_sync(0xFFFFFFFFu, trun, 31);
  if (lane == 0) {
    if (OP != kOpDw) sh.tile_start[GL] = static_cast<int32_t>(ttotal);
    sh.total_tiles = static_cast<int32_t>(ttotal);
    sh.zero_lo = sh.bound[a.group_offset];
    sh.zero_hi = sh.bound[a.group_offset + GL];
  }
}

template <int OP, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const GemmShared<PAIR>& sh, const GemmArgs& a, int t) {
  SchedView v;
  v.bound = sh.bound;
  v.tile_start = sh.tile_start;
  v.group_offset = a.group_offset;
  v.g_local = a.g_local;
  v.n_tiles = a.n_tiles;
  v.band_tiles = a.band_tiles;
  v.dw_m_tiles = a.dw_m_tiles;
  v.kc = a.kc;
  return decode_tile_view<OP, TileCfg<PAIR>::kTileM>(v, t);
}

// Zero rows [z0, z1) of one stage of a dw block in both operands: each row is
// one 128-byte line per 64-wide chunk (A chunks, then B chunks).  Then make
// the writes visible to the tensor core (async proxy).
template <int A_CHUNKS, int B_CHUNKS>
__device__ __forceinline__ void dw_zero_rows(uint8_t* a_st, uint8_t* b_st, int z0, int z1, int lane) {
  constexpr int kChunks = A_CHUNKS + B_CHUNKS;
  const int nunits = (z1 - z0) * kChunks * 8;  // 16-byte units
  for (int u = lane; u < nunits; u += 32) {
    const int row = z0 + u / (kChunks * 8);
    const int rest = u % (kChunks * 8);
    const int chunk = rest >> 3;
    const int part = rest & 7;
    uint8_t* base = chunk < A_CHUNKS ? a_st + chunk * (kBK * 128)
                                     : b_st + (chunk - A_CHUNKS) * (kBK * 128);
    *reinterpret_cast<uint4*>(base + row * 128 + part * 16) = make_uint4(0, 0, 0, 0);
  }
  ptx::fence_proxy_async_smem();
}

// Wait until *counter > value: a bounded poll on a shared-memory counter that
// another warp of the CTA advances (gives up like mbar_wait_bounded).
__device__ __forceinline__ bool wait_counter_above(const volatile int32_t* counter, int32_t value,
                                                   volatile int* abort_flag, uint64_t limit_ns) {
  if (*counter > value) return true;
  const uint64_t t0 = ptx::global_timer_ns();
#pragma unroll 1
  while (*counter <= value) {
    if (*abort_flag) return false;
    if (ptx::global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// One TMA box of a ring stage: which tensor map (A or B), its coordinates
// (innermost first) and where it lands inside the stage's A or B tile.
struct Box {
  int32_t x, y, z;
  uint32_t off;  // bytes from the start of the stage's A (or B) tile
  bool on;       // this slot carries a box
  bool b;        // tensor map B (else A)
  bool d3;       // 3-D map (else 2-D)
};

// The boxes that fill one ring stage of this CTA: K block kb of tile tl.
// Slots are fixed per configuration (compile-time indices keep the list in
// registers); unused slots have on == false.
template <int OP, bool PAIR, bool GLU>
__device__ __forceinline__ void stage_boxes(const Tile& tl, int kb, uint32_t rank, const GemmArgs& a,
                                            Box (&bx)[6]) {
  constexpr int TM = TileCfg<PAIR>::kTileM;
  constexpr uint32_t kChunk = kBK * 128;  // bytes of one 64-wide chunk of a stage tile
  auto put = [&](int i, bool on, bool b, bool d3, int32_t x, int32_t y, int32_t z, uint32_t off) {
    bx[i].x = x;
    bx[i].y = y;
    bx[i].z = z;
    bx[i].off = off;
    bx[i].on = on;
    bx[i].b = b;
    bx[i].d3 = d3;
  };
#pragma unroll
  for (int i = 0; i < 6; ++i) bx[i].on = false;
  if (OP == kOpDw) {
    // a chunked map lands its 64-column chunks 8 KB apart, as separate boxes would;
    // with group maps the rows are counted from the group's first row
    int row0;
    if (a.group_maps) dw_group_block(tl, kb, &row0);
    else row0 = dw_block_row(tl, kb);
    const int ka = tl.m_idx * TM + static_cast<int>(rank) * kBM;
    constexpr int b_cols = PAIR ? kBN / 2 : kBN;
    const int nb = tl.n_idx * kBN + static_cast<int>(rank) * b_cols;
    const bool ac = a.a_chunked != 0, bc = a.b_chunked != 0;
    put(0, true, false, ac, ac ? 0 : ka, row0, ac ? ka / 64 : 0, 0);
    put(1, !ac, false, false, ka + 64, row0, 0, kChunk);
    put(2, true, true, bc, bc ? 0 : nb, row0, bc ? nb / 64 : 0, 0);
#pragma unroll
    for (int c = 1; c < b_cols / 64; ++c) put(2 + c, !bc, true, false, nb + c * 64, row0, 0, c * kChunk);
    return;
  }
  const int arow = tl.row_load + static_cast<int>(rank) * kBM;
  put(0, true, false, false, kb * kBK, arow, 0, 0);
  if (OP == kOpFwd) {
    // rhs [g, k, n] as (n, k, g): MN-major B, 64 columns per box
    constexpr int kBoxes = PAIR ? 2 : 4;
#pragma unroll
    for (int c = 0; c < kBoxes; ++c) {
      int x;
      if (GLU) {
        // gate columns then up columns (in a pair: the even CTA gate, the odd CTA up)
        const bool up = PAIR ? rank != 0 : c >= 2;
        x = (up ? a.glu_f : 0) + tl.n_idx * (kBN / 2) + (PAIR ? c : (c & 1)) * 64;
      } else {
        x = tl.n_idx * kBN + static_cast<int>(rank) * (kBN / 2) + c * 64;
      }
      put(1 + c, true, true, true, x, kb * kBK, tl.j, c * kChunk);
    }
  } else {
    // dx: w [g, k, n] as (n, k, g): the K-major B of w^T, one box
    put(1, true, true, true, kb * kBK, tl.n_idx * kBN + static_cast<int>(rank) * (PAIR ? kBN / 2 : 0),
        tl.j, 0);
  }
}

template <int OP, int EPI, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  constexpr bool GLU = (EPI == kEpiGlu);
  static_assert(EPI != kEpiGluBwd || OP == kOpDx, "the GLU backward epilogue follows dx");
  static_assert((EPI != kEpiF32 && EPI != kEpiF32Acc) || OP == kOpDw, "f32 output is for dw");
  constexpr bool F32OUT = (EPI == kEpiF32 || EPI == kEpiF32Acc);
  using Cfg = TileCfg<PAIR>;
  constexpr int S = Cfg::kStagesN;
  constexpr int TM = Cfg::kTileM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::kStageA;
  GemmShared<PAIR>& sh = *reinterpret_cast<GemmShared<PAIR>*>(smem + S * Cfg::kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;  // 0 = the CTA that issues the MMA
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_addr(&sh.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.empty[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.efull[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.pready[s]), PAIR ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&sh.tfull[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.tempty[b]), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&sh.drain), 1);
    sh.abort_flag = 0;
    sh.fills = 0;
    sh.maps_built = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && args.kc > 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_addr(&sh.tmem_base), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&sh.tmem_base), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 2) build_schedule<OP, PAIR>(sh, args, lane);
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // the peer's barriers are initialised before any remote use
  ptx::tc_fence_after();

  const int total = sh.total_tiles;
  const uint64_t tlimit = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pend_mask = 0, pend_par = 0;  // fills whose consumption is not yet seen
      uint32_t pend_edge = 0, pend_cpar = 0;  // ... their barrier (edge or not) and its parity
      uint32_t fpar = 0, epar = 0;            // per-slot parities of full / efull
      int32_t n_fills = 0;
      bool ok = true;
      int32_t map_tiles = 0;  // dw with group maps: tiles with rows so far
      for (int t = unit; t < total && ok; t += units) {
        const Tile tl = decode_tile<OP, PAIR>(sh, args, t);
        const CUtensorMap* map_a = &tmap_a;
        const CUtensorMap* map_b = &tmap_b;
        if (OP == kOpDw && args.group_maps && tl.nkb > 0) {
          // this tile's maps (rebased to its group by the map warp): wait until they
          // are published, then acquire them for the copies
          if (!wait_counter_above(&sh.maps_built, map_tiles, abort_flag, tlimit)) {
            ok = false;
            break;
          }
          map_a = args.maps + (static_cast<size_t>(blockIdx.x) * kMapSlots + map_tiles % kMapSlots) * 2;
          map_b = map_a + 1;
          ptx::tmap_acquire(map_a);
          ptx::tmap_acquire(map_b);
          ++map_tiles;
        }
        for (int kb = 0; kb < tl.nkb; ++kb) {
          // Everything this fill needs is worked out before waiting for its slot, so
          // that the copies go out as soon as the slot is free (with the operands
          // arriving just in time, any work between the two adds to every block).
          const uint32_t fb_local = ptx::smem_addr(&sh.full[stage]);
          const uint32_t a_dst = ptx::smem_addr(sA + stage * Cfg::kStageA);
          const uint32_t b_dst = ptx::smem_addr(sB + stage * Cfg::kStageB);
          // dw: the last block of a group whose start straddles a 16-row K step must be
          // zeroed in each CTA before the MMA reads it.  Its copy counts on this CTA's
          // own edge barrier (efull), which only edge blocks use; the edge warp waits
          // there, zeroes, and signals the MMA.
          bool edge = false;
          if (OP == kOpDw && !args.group_maps) {
            int z0, z1;
            dw_edge(tl, kb, z0, z1);
            edge = z1 > z0;
          }
          const uint32_t eb_local = ptx::smem_addr(&sh.efull[stage]);
          // Non-edge fills of both CTAs of a pair count on the even CTA's barrier, which
          // expects them all; the odd CTA's copies may land before that expectation is
          // posted (the phase cannot complete before the even CTA's arrival).
          const uint32_t fb = edge ? eb_local : (PAIR ? ptx::map_to_rank(fb_local, 0) : fb_local);
          Box bx[6];
          stage_boxes<OP, PAIR, GLU>(tl, kb, rank, args, bx);
          if (!ptx::mbar_wait_bounded(ptx::smem_addr(&sh.empty[stage]), phase ^ 1,
                                              abort_flag, tlimit)) {
            ok = false;
            break;
          }
          pend_mask &= ~(1u << stage);
          if (!PAIR || edge) ptx::mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          else if (rank == 0) ptx::mbar_arrive_expect_tx(fb_local, 2 * Cfg::kStageBytes);
#pragma unroll
          for (int i = 0; i < 6; ++i) {
            if (!bx[i].on) continue;
            const uint32_t dst = (bx[i].b ? b_dst : a_dst) + bx[i].off;
            const CUtensorMap* map = bx[i].b ? map_b : map_a;
            if (PAIR) {
              if (bx[i].d3) ptx::tma_load_3d_pair(dst, map, fb, bx[i].x, bx[i].y, bx[i].z);
              else ptx::tma_load_2d_pair(dst, map, fb, bx[i].x, bx[i].y);
            } else {
              if (bx[i].d3) ptx::tma_load_3d(dst, map, fb, bx[i].x, bx[i].y, bx[i].z);
              else ptx::tma_load_2d(dst, map, fb, bx[i].x, bx[i].y);
            }
          }
          pend_mask |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          // parity of the barrier this fill completes (full: non-edge fills, efull: edge fills)
          const uint32_t cnt_par = edge ? ((epar >> stage) & 1u) : ((fpar >> stage) & 1u);
          pend_edge = (pend_edge & ~(1u << stage)) | ((edge ? 1u : 0u) << stage);
          pend_cpar = (pend_cpar & ~(1u << stage)) | (cnt_par << stage);
          if (edge) epar ^= 1u << stage; else fpar ^= 1u << stage;
          *reinterpret_cast<volatile int32_t*>(&sh.fills) = ++n_fills;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Wait until every fill of this CTA's ring has been consumed, so that no MMA
      // commit (possibly from the peer CTA) arrives on a barrier after this CTA exits.
      // On abort, wait (bounded) for the copies still in flight instead; the odd CTA
      // of a pair cannot observe its copies (they count on the even CTA's barrier),
      // so it gives them a fixed grace period.
      volatile int no_abort = 0;
      for (int s = 0; s < S; ++s) {
        if (!(pend_mask & (1u << s))) continue;
        const uint32_t par = (pend_par >> s) & 1u;
        if (*abort_flag) {
          const bool e = (pend_edge >> s) & 1u;
          const uint32_t cp = (pend_cpar >> s) & 1u;
          if (e)
            ptx::mbar_wait_bounded(ptx::smem_addr(&sh.efull[s]), cp, &no_abort, kDrainNs);
          else if (!PAIR || rank == 0)
            ptx::mbar_wait_bounded(ptx::smem_addr(&sh.full[s]), cp, &no_abort, kDrainNs);
        } else {
          ptx::mbar_wait_bounded(ptx::smem_addr(&sh.empty[s]), par, &no_abort, kDrainNs);
        }
      }
      if (PAIR && rank != 0 && *abort_flag && (pend_mask & ~pend_edge) != 0) {
        const uint64_t t0 = ptx::global_timer_ns();
        while (ptx::global_timer_ns() - t0 < kGraceNs) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread does all of it: waits, issue and commits.  (Waiting with the
    // whole warp and voting on the result cost ~100 ns per K block, during which
    // the tensor pipe ran dry.)
    if ((!PAIR || rank == 0) && lane == 0) {
      constexpr bool a_mn = (OP == kOpDw);
      constexpr bool b_mn = (OP != kOpDx);
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(TM, kBN, a_mn, b_mn);
      constexpr uint32_t b_lbo = kBK * 128;  // MN-major B: stride between 64-wide chunks
      int stage = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t pready_par = 0;  // per-slot parity of pready (edge blocks)
      uint32_t full_par = 0;    // per-slot parity of full (every other block)
      bool ok = true;
      for (int t = unit; t < total && ok; t += units) {
        const Tile tl = decode_tile<OP, PAIR>(sh, args, t);
        if (tl.nkb == 0) continue;
        ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.tempty[acc]), acc_phase ^ 1, abort_flag,
                                    tlimit);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = sh.tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < tl.nkb; ++kb) {
          int kk0 = 0;  // first 16-deep K step issued for this block
          bool edge = false;
          if (OP == kOpDw) {
            if (args.group_maps) {
              // the first block's rows above the group arrived as zeros: skip their
              // whole 16-row steps
              int row;
              kk0 = dw_group_block(tl, kb, &row);
            } else {
              int z0, z1;
              kk0 = dw_edge(tl, kb, z0, z1);
              edge = z1 > z0;
            }
          }
          // the block's operand descriptors, worked out before its wait (as the
          // producer does for its copies) so that the MMAs issue as soon as it lands
          const uint32_t a_addr = ptx::smem_addr(sA + stage * Cfg::kStageA);
          const uint32_t b_addr = ptx::smem_addr(sB + stage * Cfg::kStageB);
          auto a_desc = [&](int kk) {
            return a_mn ? ptx::sw128_desc(a_addr + kk * 2048, kBK * 128, 1024)
                        : ptx::sw128_desc(a_addr + kk * 32, 16, 1024);
          };
          auto b_desc = [&](int kk) {
            return b_mn ? ptx::sw128_desc(b_addr + kk * 2048, b_lbo, 1024)
                        : ptx::sw128_desc(b_addr + kk * 32, 16, 1024);
          };
          uint64_t ad[kBK / 16], bd[kBK / 16];
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            ad[kk] = a_desc(kk);
            bd[kk] = b_desc(kk);
          }
          if (edge) {
            // rows of a neighbouring group (or a NaN) must not enter the sum: the
            // straddling rows of an edge block are zeroed by the edge warp of each CTA,
            // which signals pready once its part is done (its copy has landed by then)
            const uint32_t pb = ptx::smem_addr(&sh.pready[stage]);
            const uint32_t par = (pready_par >> stage) & 1u;
            ok = PAIR ? ptx::mbar_wait_bounded_cluster(pb, par, abort_flag, tlimit)
                      : ptx::mbar_wait_bounded(pb, par, abort_flag, tlimit);
            pready_par ^= 1u << stage;
          } else {
            ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.full[stage]), (full_par >> stage) & 1u,
                                        abort_flag, tlimit);
            full_par ^= 1u << stage;
          }
          if (!ok) break;
          ptx::tc_fence_after();
          auto mma = [&](uint64_t adesc, uint64_t bdesc, uint32_t accum) {
            if (PAIR) ptx::tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, accum);
            else ptx::tc_mma_bf16(d_tmem, adesc, bdesc, idesc, accum);
          };
          if (kk0 == 0) {
            // every block but a dw group's straddling last one: four MMAs back to
            // back (with a skip test in front of each, dw's issue took ~1.3x as long)
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) mma(ad[kk], bd[kk], (kb > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll 1
            for (int kk = kk0; kk < kBK / 16; ++kk)
              mma(a_desc(kk), b_desc(kk), (kb > 0 || kk > kk0) ? 1u : 0u);
          }
          if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&sh.empty[stage]), 0x3);
          else ptx::tc_commit(ptx::smem_addr(&sh.empty[stage]));
          if (++stage == S) stage = 0;
        }
        if (!ok) break;
        if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&sh.tfull[acc]), 0x3);
        else ptx::tc_commit(ptx::smem_addr(&sh.tfull[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (*abort_flag) {
        // wait until every MMA this thread issued has completed before TMEM is freed
        volatile int no_abort = 0;
        if (PAIR) ptx::tc_commit_pair(ptx::smem_addr(&sh.drain), 0x1);
        else ptx::tc_commit(ptx::smem_addr(&sh.drain));
        ptx::mbar_wait_bounded(ptx::smem_addr(&sh.drain), 0, &no_abort, kDrainNs);
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Eight warps, two per 32-lane quarter of the accumulator (32 tile rows);
    // the two split the tile's 32-column chunks.  A chunk is read from TMEM
    // (thread = row), rounded to bf16 (or put through the GLU forward or
    // backward), transposed through a 2 KB XOR-swizzled staging buffer, and
    // stored 8 rows x 64 contiguous bytes per instruction.
    const int e = warp - 2;
    const int q = warp & 3;      // TMEM lane quarter this warp may access
    const int half = e >> 2;     // which half of the chunks
    constexpr int tile_w = GLU ? kBN / 2 : kBN;
    constexpr int kChunks = tile_w / 32;
    const int c_begin = half * (kChunks / 2), c_end = c_begin + kChunks / 2;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
    uint4* stg = sh.epi[e];
    const uint32_t tempty_leader =
        PAIR ? ptx::map_to_rank(ptx::smem_addr(&sh.tempty[0]), 0) : 0u;
    const int sr = lane >> 2;      // row (within 8) this lane stores
    const int piece = lane & 3;    // 16-byte piece of the row's 64 bytes
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = unit; t < total; t += units) {
      const Tile tl = decode_tile<OP, PAIR>(sh, args, t);
      // first row of this warp's 32 rows and the rows it may write: [lo, hi)
      const int wrow0 = (OP == kOpDw ? tl.m_idx * TM : tl.row_load) +
                        static_cast<int>(rank) * kBM + q * 32;
      const int lo = OP == kOpDw ? 0 : tile_store_lo(tl, TM);
      const int hi = OP == kOpDw ? args.m_out : tile_store_hi(tl);
      __nv_bfloat16* base =
          OP == kOpDw ? out + static_cast<size_t>(tl.j) * args.m_out * args.ldo : out;
      const int col0 = tl.n_idx * tile_w;
      // write the 16 packed words of this lane's row into the staging buffer, then
      // store the chunk's 32 rows x 32 columns to global memory
      // (col_off shifts the destination, e.g. to the d_up half of a fused row)
      auto emit = [&](const uint32_t (&p)[16], int col, int col_off) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          stg[lane * 4 + (v ^ ((lane >> 1) & 3))] =
              make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rl = it * 8 + sr;
          const uint4 val = stg[rl * 4 + (piece ^ ((rl >> 1) & 3))];
          const int row = wrow0 + rl;
          const int c = col + piece * 8;
          if (row >= lo && row < hi && c + 8 <= args.n_out)
            *reinterpret_cast<uint4*>(base + static_cast<size_t>(row) * args.ldo + col_off + c) = val;
        }
        __syncwarp();
      };
      // f32 output of dw, 16 columns (64 bytes a row) at a time through the same
      // staging layout; the accumulating form adds them to what the output holds
      auto emit_f32 = [&](const uint32_t* v16, int col) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          stg[lane * 4 + (v ^ ((lane >> 1) & 3))] =
              make_uint4(v16[4 * v], v16[4 * v + 1], v16[4 * v + 2], v16[4 * v + 3]);
        __syncwarp();
        float* outf = reinterpret_cast<float*>(args.out) +
                      static_cast<size_t>(tl.j) * args.m_out * args.ldo;
        // the accumulating form reads the prior values of all four rows before it
        // writes any (one read-modify-write after another serialised four HBM
        // round trips)
        uint4 prior[4];
        if (EPI == kEpiF32Acc) {
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int row = wrow0 + it * 8 + sr;
            const int c = col + piece * 4;
            prior[it] = (row < hi && c + 4 <= args.n_out)
                            ? *reinterpret_cast<const uint4*>(outf + static_cast<size_t>(row) * args.ldo + c)
                            : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int rl = it * 8 + sr;
          uint4 val = stg[rl * 4 + (piece ^ ((rl >> 1) & 3))];
          const int row = wrow0 + rl;
          const int c = col + piece * 4;
          if (row < hi && c + 4 <= args.n_out) {
            uint4* dst = reinterpret_cast<uint4*>(outf + static_cast<size_t>(row) * args.ldo + c);
            if (EPI == kEpiF32Acc) {
              const uint4 o = prior[it];
              val = make_uint4(__float_as_uint(__fadd_rn(__uint_as_float(o.x), __uint_as_float(val.x))),
                               __float_as_uint(__fadd_rn(__uint_as_float(o.y), __uint_as_float(val.y))),
                               __float_as_uint(__fadd_rn(__uint_as_float(o.z), __uint_as_float(val.z))),
                               __float_as_uint(__fadd_rn(__uint_as_float(o.w), __uint_as_float(val.w))));
            }
            *dst = val;
          }
        }
        __syncwarp();
      };
      if (tl.nkb == 0) {
        const uint32_t z[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        for (int c = c_begin; c < c_end; ++c) {
          if (F32OUT) {
            if (EPI == kEpiF32) {  // an empty group's block is zero (accumulating: unchanged)
              emit_f32(z, col0 + c * 32);
              emit_f32(z, col0 + c * 32 + 16);
            }
          } else {
            emit(z, col0 + c * 32, 0);
            if (EPI == kEpiGluBwd) emit(z, col0 + c * 32, args.n_out);
          }
        }
        continue;
      }
      if (EPI == kEpiF32Acc) {
        // the prior values this lane will add to (its row, this warp's columns) do not
        // depend on the accumulator: bring them into L2 while the MMAs run
        const int row = wrow0 + lane;
        if (row < hi) {
          const float* rp = reinterpret_cast<const float*>(args.out) +
                            (static_cast<size_t>(tl.j) * args.m_out + row) * args.ldo;
#pragma unroll
          for (int c = c_begin * 32; c < c_end * 32; c += 32)  // 32 floats = 128 bytes
            if (col0 + c < args.n_out) ptx::prefetch_l2(rp + col0 + c);
        }
      }
      bool ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.tfull[acc]), acc_phase, abort_flag,
                                       tlimit);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tbase =
          sh.tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      if (GLU) {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          uint32_t g[32], u[32], p[16];
          ptx::tmem_load_32cols(tbase + c * 32, g);
          ptx::tmem_load_32cols(tbase + kBN / 2 + c * 32, u);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(glu_fwd_fast(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                               glu_fwd_fast(__uint_as_float(g[2 * i + 1]),
                                            __uint_as_float(u[2 * i + 1])));
          emit(p, col0 + c * 32, 0);
        }
      } else if (EPI == kEpiGluBwd) {
        // dh (f32, this tile's accumulator) meets the saved gate / up of the same row:
        // each thread reads its row's 32 gate and 32 up values, the backward of the
        // GLU runs per element in f32, and [d_gate | d_up] leave through emit().
        const __nv_bfloat16* fused = reinterpret_cast<const __nv_bfloat16*>(args.aux);
        const int row = wrow0 + lane;
        const bool row_ok = row >= lo && row < hi;
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          const int col = col0 + c * 32;
          uint4 G[4], U[4];
          const __nv_bfloat16* src = fused + static_cast<size_t>(row) * (2 * args.n_out) + col;
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            if (row_ok && col + 8 * w4 + 8 <= args.n_out) {
              G[w4] = __ldg(reinterpret_cast<const uint4*>(src) + w4);
              U[w4] = __ldg(reinterpret_cast<const uint4*>(src + args.n_out) + w4);
            } else {
              G[w4] = make_uint4(0, 0, 0, 0);
              U[w4] = make_uint4(0, 0, 0, 0);
            }
          }
          uint32_t v[32], pg[16], pu[16];
          ptx::tmem_load_32cols(tbase + c * 32, v);
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            const uint32_t gw[4] = {G[w4].x, G[w4].y, G[w4].z, G[w4].w};
            const uint32_t uw[4] = {U[w4].x, U[w4].y, U[w4].z, U[w4].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float dg0, du0, dg1, du1;
              glu_bwd_fast(bf16_lo(gw[i]), bf16_lo(uw[i]), __uint_as_float(v[w4 * 8 + 2 * i]), dg0,
                           du0);
              glu_bwd_fast(bf16_hi(gw[i]), bf16_hi(uw[i]), __uint_as_float(v[w4 * 8 + 2 * i + 1]), dg1,
                           du1);
              pg[w4 * 4 + i] = bf16x2_neg_zero_to_pos(pack_bf16x2(dg0, dg1));
              pu[w4 * 4 + i] = bf16x2_neg_zero_to_pos(pack_bf16x2(du0, du1));
            }
          }
          emit(pg, col, 0);
          emit(pu, col, args.n_out);
        }
      } else if (F32OUT) {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          uint32_t v[32];
          ptx::tmem_load_32cols(tbase + c * 32, v);
          emit_f32(v, col0 + c * 32);
          emit_f32(v + 16, col0 + c * 32 + 16);
        }
      } else {
#pragma unroll 1
        for (int c = c_begin; c < c_end; ++c) {
          uint32_t v[32], p[16];
          ptx::tmem_load_32cols(tbase + c * 32, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          emit(p, col0 + c * 32, 0);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && rank != 0)
          ptx::mbar_arrive_cluster(tempty_leader + static_cast<uint32_t>(acc * sizeof(uint64_t)));
        else
          ptx::mbar_arrive(ptx::smem_addr(&sh.tempty[acc]));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else if (OP == kOpDw && warp == 2 + kEpiWarps && args.group_maps) {
    // ------------------------------------------------------------ dw group maps
    // For each of this CTA's tiles with rows, rebase copies of the x and y maps to
    // the tile's group (address = the group's first row, rows = the group's rows)
    // and publish them to the CTA's next map slot, ahead of the producer.  Rows
    // outside the group are then out of bounds for the copies and land as zeros,
    // so no block needs zeroing.  A slot is rewritten only once the producer has
    // filled a whole ring beyond the last block read through it, i.e. once every
    // copy through its previous maps has landed.
    const uint32_t st_a = ptx::smem_addr(sh.mapstage[0]);
    const uint32_t st_b = ptx::smem_addr(sh.mapstage[1]);
    const uint4* src_a = reinterpret_cast<const uint4*>(&tmap_a);
    const uint4* src_b = reinterpret_cast<const uint4*>(&tmap_b);
    int64_t fills_end[kMapSlots];  // per slot: producer fills through its last tile
    int64_t fills = 0;
    int32_t built = 0;
    bool ok = true;
    for (int t = unit; t < total && ok; t += units) {
      const Tile tl = decode_tile<OP, PAIR>(sh, args, t);
      fills += tl.nkb;
      if (tl.nkb == 0) continue;
      const int slot = built % kMapSlots;
      if (built >= kMapSlots) {
        ok = wait_counter_above(&sh.fills, static_cast<int32_t>(fills_end[slot] + S - 1), abort_flag,
                                tlimit);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
      }
      if (lane < 8) reinterpret_cast<uint4*>(sh.mapstage[0])[lane] = src_a[lane];
      else if (lane < 16) reinterpret_cast<uint4*>(sh.mapstage[1])[lane - 8] = src_b[lane - 8];
      __syncwarp();
      if (lane == 0) {
        const uint32_t rows = static_cast<uint32_t>(tl.re - tl.rs);
        ptx::tmap_replace_address(st_a, static_cast<const char*>(args.x_base) +
                                            static_cast<int64_t>(tl.rs) * args.x_row_bytes);
        ptx::tmap_replace_dim1(st_a, rows);
        ptx::tmap_replace_address(st_b, static_cast<const char*>(args.y_base) +
                                            static_cast<int64_t>(tl.rs) * args.y_row_bytes);
        ptx::tmap_replace_dim1(st_b, rows);
      }
      __syncwarp();
      CUtensorMap* dst = args.maps + (static_cast<size_t>(blockIdx.x) * kMapSlots + slot) * 2;
      ptx::tmap_publish(dst, st_a);
      ptx::tmap_publish(dst + 1, st_b);
      fills_end[slot] = fills;
      ++built;
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int32_t*>(&sh.maps_built) = built;
      }
    }
  } else if (OP == kOpDw && warp == 2 + kEpiWarps) {
    // ------------------------------------------------------------ dw edge rows
    // For each edge block (the last K block of a group, whose first rows precede
    // the group), wait for this CTA's own copy, zero the rows of the straddling
    // 16-row step in both operands, and signal the MMA (in a pair: the even
    // CTA's barrier, which expects both CTAs).  The producer runs ahead of the
    // MMA, so this usually finishes before the MMA reaches the block.
    int stage = 0;
    uint32_t lpar = 0;  // per-slot parity of this CTA's efull barrier
    const uint32_t pready0 = PAIR ? ptx::map_to_rank(ptx::smem_addr(&sh.pready[0]), 0)
                                  : ptx::smem_addr(&sh.pready[0]);
    bool ok = true;
    for (int t = unit; t < total && ok; t += units) {
      const Tile tl = decode_tile<OP, PAIR>(sh, args, t);
      for (int kb = 0; kb < tl.nkb; ++kb) {
        int z0, z1;
        dw_edge(tl, kb, z0, z1);
        if (z1 > z0) {
          ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.efull[stage]), (lpar >> stage) & 1u,
                                      abort_flag, tlimit);
          lpar ^= 1u << stage;
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          dw_zero_rows<2, Cfg::kBCols / 64>(sA + stage * Cfg::kStageA, sB + stage * Cfg::kStageB,
                                           z0, z1, lane);
          __syncwarp();
          if (lane == 0) {
            const uint32_t pb = pready0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
            if (PAIR) ptx::mbar_arrive_cluster(pb);
            else ptx::mbar_arrive(pb);
          }
        }
        if (++stage == S) stage = 0;
      }
    }
  } else if (OP != kOpDw && warp == 2 + kEpiWarps) {
    // ------------------------------------------------------------ zero fill
    // Rows [0, zero_lo) and [zero_hi, L) are two contiguous byte ranges of the
    // output (its rows are contiguous).  Each CTA takes a contiguous 16-byte
    // aligned share of their concatenation and has the bulk-copy engine write it
    // from a 4 KB zero block in shared memory.  Units (CTAs or CTA pairs) with
    // one tile fewer than the others take twice the share: they have a tile's
    // time to spare at the end.  The writes are paced by the CTA's own progress
    // (the bytes issued follow the stages its producer has filled), so that they
    // spread over the run instead of meeting the operand reads in HBM in one burst.
    for (int i = lane; i < 256; i += 32) sh.zeros[i] = make_uint4(0, 0, 0, 0);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const uint64_t row_bytes = static_cast<uint64_t>(args.ldo) * 2;
      const uint64_t lo_bytes = static_cast<uint64_t>(sh.zero_lo) * row_bytes;
      const uint64_t z_bytes = lo_bytes + static_cast<uint64_t>(sh.L - sh.zero_hi) * row_bytes;
      const uint64_t units16 = z_bytes / 16;
      uint64_t u0, u1;
      zero_share(units16, unit, units, total, PAIR, PAIR ? static_cast<int>(blockIdx.x & 1u) : 0,
                 u0, u1);
      if (u1 > u0) {
        int64_t stages = 0;  // stages this CTA's producer fills in all
        for (int t = unit; t < total; t += units) stages += decode_tile<OP, PAIR>(sh, args, t).nkb;
        const uint64_t share = u1 - u0;
        const volatile int32_t* fills = &sh.fills;
        char* base = reinterpret_cast<char*>(args.out);
        const uint32_t src = ptx::smem_addr(sh.zeros);
        uint64_t done = 0;  // 16-byte units issued
        uint64_t t_last = ptx::global_timer_ns();
#pragma unroll 1
        while (done < share) {
          const int64_t f = *fills;
          // dx (the fused GLU backward: zero rows twice as wide, a shorter GEMM)
          // runs its zeros twice as fast as its stages, so that they are out
          // before the CTA's last epilogues; the forward keeps them in step
          constexpr uint64_t kLead = OP == kOpFwd ? 1 : 2;
          uint64_t target = (stages == 0 || f >= stages)
                                ? share
                                : share * static_cast<uint64_t>(f) * kLead / static_cast<uint64_t>(stages);
          if (target > share) target = share;
          if (target <= done) {
            // pacing only: give up (and unwind with the CTA) like any other wait
            if (*abort_flag) break;
            if (ptx::global_timer_ns() - t_last > tlimit) {
              *abort_flag = 1;
              break;
            }
            __nanosleep(500);
            continue;
          }
          uint64_t b = (u0 + done) * 16;
          const uint64_t b1 = (u0 + target) * 16;
          while (b < b1) {
            const bool low = b < lo_bytes;
            const uint64_t seg_end = low ? lo_bytes : z_bytes;
            const uint64_t addr = low ? b : static_cast<uint64_t>(sh.zero_hi) * row_bytes + (b - lo_bytes);
            uint64_t len = (b1 < seg_end ? b1 : seg_end) - b;
            if (len > 4096) len = 4096;
            ptx::bulk_copy_s2g(base + addr, src, static_cast<uint32_t>(len));
            b += len;
          }
          ptx::bulk_commit();
          done = target;
          t_last = ptx::global_timer_ns();
        }
        ptx::bulk_wait_read_all();
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // the peer no longer touches this CTA's barriers or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR) ptx::tmem_dealloc_pair(sh.tmem_base, kTmemCols);
    else ptx::tmem_dealloc(sh.tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && sh.abort_flag && args.status != nullptr)
    atomicOr(args.status, RD_STATUS_TIMEOUT);
}

template <int OP, int EPI, bool PAIR>
cudaError_t launch_gemm_impl(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                             const GemmArgs& args, int grid, cudaStream_t stream) {
  constexpr size_t smem = gemm_smem_bytes_t<PAIR>();
  // the shared-memory size attribute is set once per device (it is per-device
  // state); two threads racing here both set it, which is harmless
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    const cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<OP, EPI, PAIR>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  if (!PAIR) {
    grouped_gemm_kernel<OP, EPI, PAIR><<<grid, kThreads, smem, stream>>>(tmap_a, tmap_b, args);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // A persistent grid must not exceed the clusters that can be resident at once:
  // a CTA pair must sit in one GPC, so fewer than (#SMs / 2) pairs may fit.  The
  // limit is queried once per device (it depends only on the kernel and the GPU).
  static std::atomic<int> max_clusters[64];
  int clusters = max_clusters[dev].load(std::memory_order_acquire);
  if (clusters == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<OP, EPI, PAIR>, &cfg);
    if (e != cudaSuccess) return e;
    clusters = n > 0 ? n : 1;
    max_clusters[dev].store(clusters, std::memory_order_release);
  }
  if (grid > 2 * clusters) grid = 2 * clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<OP, EPI, PAIR>, tmap_a, tmap_b, args);
}

}  // namespace rd
