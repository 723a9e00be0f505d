// unsort.cu -- valid-rows unsort backward: for every row r < L of the packed
// buffer, grad[r, :] = bf16(f32(g[r, :]) * w[r]) and the f32 routing-weight
// row dot dot[r] = sum_c f32(g[r, c]) * f32(y[r, c]).
//
// MaxText PR #5760 ("MoE wo FSDP sharding and valid-rows-only MoE kernels",
// commit message, kernels/ragged/unsort_bwd_rows.py; review comment on the
// race of concurrent blocks updating one row's dot).  Here one warp owns a
// whole row: it streams the row in 16-byte vectors, writes the weighted
// gradient and reduces the dot in registers and shuffles, so no two CTAs ever
// touch the same output and no partial sums go through memory.  Rows at or
// past L are neither read nor written.  HBM-bound: 4 bytes read and 2 written
// per element, plus 8 bytes per row.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_args.h"
#include "glu_math.cuh"

namespace rd {
namespace {

constexpr int kUnsortThreads = 256;
constexpr int kUnsortWarps = kUnsortThreads / 32;
constexpr int kUnsortBatch = 4;  // 16-byte vectors per lane in flight

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// two bf16 of g times w (one f32 multiply each, one bf16 rounding); the dot
// accumulates the exact f32 products of g and y
__device__ __forceinline__ uint32_t scale2(uint32_t g, uint32_t y, float w, float& dot) {
  const float g0 = bf16_lo(g), g1 = bf16_hi(g);
  dot = __fadd_rn(dot, __fmul_rn(g0, bf16_lo(y)));
  dot = __fadd_rn(dot, __fmul_rn(g1, bf16_hi(y)));
  return pack_bf16x2(__fmul_rn(g0, w), __fmul_rn(g1, w));
}

__global__ void __launch_bounds__(kUnsortThreads)
    unsort_bwd_rows_kernel(const uint4* __restrict__ g, const uint4* __restrict__ y,
                           const float* __restrict__ w, uint4* __restrict__ grad,
                           float* __restrict__ dot, int32_t rows, int32_t hidden,
                           const int32_t* limit) {
  int32_t L = rows;
  if (limit != nullptr) {
    const int32_t v = *limit;
    L = v < 0 ? 0 : (v > rows ? rows : v);
  }
  const int vpr = hidden >> 3;
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * kUnsortWarps;
  for (int r = blockIdx.x * kUnsortWarps + (threadIdx.x >> 5); r < L; r += stride) {
    const uint4* g_row = g + static_cast<size_t>(r) * vpr;
    const uint4* y_row = y + static_cast<size_t>(r) * vpr;
    uint4* o_row = grad + static_cast<size_t>(r) * vpr;
    const float wr = w[r];
    float acc = 0.0f;
    for (int v0 = lane; v0 < vpr; v0 += 32 * kUnsortBatch) {
      uint4 gv[kUnsortBatch], yv[kUnsortBatch];
#pragma unroll
      for (int b = 0; b < kUnsortBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr) {
          gv[b] = ld_stream(g_row + v);
          yv[b] = ld_stream(y_row + v);
        }
      }
#pragma unroll
      for (int b = 0; b < kUnsortBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr)
          o_row[v] = make_uint4(scale2(gv[b].x, yv[b].x, wr, acc), scale2(gv[b].y, yv[b].y, wr, acc),
                                scale2(gv[b].z, yv[b].z, wr, acc), scale2(gv[b].w, yv[b].w, wr, acc));
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, d));
    if (lane == 0) dot[r] = acc;
  }
}

}  // namespace

cudaError_t launch_unsort_bwd_rows(const void* g, const void* y, const float* w, void* grad,
                                   float* dot, int32_t rows, int32_t hidden, const int32_t* limit,
                                   int grid, cudaStream_t stream) {
  unsort_bwd_rows_kernel<<<grid, kUnsortThreads, 0, stream>>>(
      static_cast<const uint4*>(g), static_cast<const uint4*>(y), w, static_cast<uint4*>(grad), dot,
      rows, hidden, limit);
  return cudaGetLastError();
}

}  // namespace rd
