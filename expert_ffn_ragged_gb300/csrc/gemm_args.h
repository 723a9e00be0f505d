// gemm_args.h -- launch arguments of the grouped-GEMM kernels (host and
// device), the tile shape, and the host-side launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "schedule.h"

namespace rd {

// What the epilogue does with the f32 accumulator.
enum GemmEpi : int {
  kEpiNone = 0,   // round to bf16 and store
  kEpiGlu = 1,    // forward: silu(gate) * up from the gate / up halves of the tile
  kEpiGluBwd = 2,  // dx of the down projection: [d_gate | d_up] from dh and the saved [gate | up]
  kEpiF32 = 3,     // dw: store the f32 accumulator as is
  kEpiF32Acc = 4   // dw: add the f32 accumulator to the f32 output already in memory
};

// UMMA tile: kBM x kBN (128 x 256) f32 accumulator per CTA, kBK (64) deep K
// blocks -- one 128-byte swizzle atom of bf16 (schedule.h).
constexpr int kEpiWarps = 8;    // two epilogue warps per 32-lane quarter of the accumulator
// 12 warps: warp 0 TMA producer, warp 1 MMA issuer, warps 2-9 epilogue (warp % 4
// is the TMEM lane quarter a warp may read, so warps 2..9 cover each quarter
// twice), warp 10 zero fill (forward / dx) or dw edge rows.  Warp 11 takes no
// role: it only joins the block-wide barriers, keeping the block at three
// whole warpgroups.
constexpr int kThreads = 384;
constexpr int kTmemCols = 2 * kBN;  // two accumulators (double buffer)
constexpr int kMaxGroups = 1024;

struct GemmArgs {
  const int32_t* group_sizes;  // [g_total], device
  const int32_t* limit;        // device scalar or null
  int32_t* status;             // device or null
  void* out;                   // bf16 output
  const void* aux;             // kEpiGluBwd: the saved fused [gate | up] buffer [m, 2 * n_out]
  int64_t ldo;                 // row stride of out (elements)
  int32_t zero_cols;           // columns of a zero row (n_out, or 2 * n_out for kEpiGluBwd)
  int32_t m;                   // token rows
  int32_t kc;                  // contraction length (fwd: k, dx: n); dw: unused (rows of each group)
  int32_t n_out;               // output width (columns stored)
  int32_t m_out;               // dw: rows of each weight block (= k)
  int32_t g_total;
  int32_t group_offset;
  int32_t g_local;
  int32_t glu_f;               // fwd with GLU: first column of the up half in rhs (= n / 2)
  int32_t n_tiles;             // output column tiles
  int32_t dw_m_tiles;          // dw: 128-row tiles of each weight block
  int32_t band_tiles;          // fwd/dx: m-tiles per band of the tile order (lhs rows kept in L2)
  int32_t a_chunked;           // dw: tmap_a is (64, rows, width / 64): one box per stage
  int32_t b_chunked;           // dw: tmap_b likewise (else 2-D maps, one box per 64 columns)
  // dw with per-group tensor maps (group_maps != 0): the CTA builds the maps of
  // its tiles' groups from tmap_a / tmap_b into its slots of `maps` (kMapSlots
  // pairs a CTA, global memory), rebasing them to each group's first row
  int32_t group_maps;
  const void* x_base;          // dw: x (the A operand) and y (the B operand)
  const void* y_base;
  int64_t x_row_bytes;
  int64_t y_row_bytes;
  CUtensorMap* maps;           // [grid][kMapSlots][2]
  uint64_t timeout_ns;         // bound of every wait inside the kernel
};

// Per-group tensor-map slots of one CTA (a ring: slot i % kMapSlots serves the
// CTA's i-th tile with rows).  It is longer than the operand ring, so a slot
// is rewritten only after every copy through its previous maps has landed.
constexpr int kMapSlots = 8;
constexpr size_t kMapBytesPerCta = static_cast<size_t>(kMapSlots) * 2 * 128;

// `pair`: the CTA-pair variant (clusters of two CTAs, 256-row tiles); `grid`
// must then be even.
cudaError_t launch_gemm_fwd(bool glu, bool pair, const CUtensorMap& tmap_a,
                            const CUtensorMap& tmap_b, const GemmArgs& args, int grid,
                            cudaStream_t stream);
cudaError_t launch_gemm_dx(bool pair, bool glu_bwd, const CUtensorMap& tmap_a,
                           const CUtensorMap& tmap_b, const GemmArgs& args, int grid,
                           cudaStream_t stream);
cudaError_t launch_gemm_dw(bool pair, int epi, const CUtensorMap& tmap_a,
                           const CUtensorMap& tmap_b, const GemmArgs& args, int grid,
                           cudaStream_t stream);

cudaError_t launch_glu_fwd(const void* fused, void* out, int32_t rows, int32_t f,
                           const int32_t* limit, int grid, cudaStream_t stream);
cudaError_t launch_glu_bwd(const void* fused, const void* d_out, void* d_fused, int32_t rows,
                           int32_t f, const int32_t* limit, int grid, cudaStream_t stream);

cudaError_t launch_unsort_bwd_rows(const void* g, const void* y, const float* w, void* grad,
                                   float* dot, int32_t rows, int32_t hidden, const int32_t* limit,
                                   int grid, cudaStream_t stream);

}  // namespace rd
