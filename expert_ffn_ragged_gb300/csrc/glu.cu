// glu.cu -- standalone SiLU-GLU forward and backward over the valid rows of
// a fused [gate | up] buffer.
//
// MaxText PR #5760 ("MoE wo FSDP sharding and valid-rows-only MoE kernels",
// commit message, kernels/ragged/glu_rows.py): silu(gate) * up over rows
// [0, limit) only, gate and up read in place from the fused buffer; the
// backward recomputes the forward and writes [d_gate | d_up] in one pass with
// the -0 -> +0 fix.  The arithmetic is in glu_math.cuh (the two-sided
// logistic with the op sequence's results wherever those are special).
//
// Both kernels are HBM-bound streams: one warp per row, 16-byte vector loads
// that bypass L1, several vectors per lane in flight before the math.
// The row count L is read on the device, so no host round trip is needed and
// the launch shape depends only on host-known sizes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_args.h"
#include "glu_math.cuh"

namespace rd {
namespace {

constexpr int kGluThreads = 256;
constexpr int kGluWarps = kGluThreads / 32;
constexpr int kFwdBatch = 4;  // 16-byte vectors per lane in flight before the math
constexpr int kBwdBatch = 2;  // the backward holds three inputs per vector

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t glu2(uint32_t g, uint32_t u) {
  return pack_bf16x2(glu_fwd_seq(bf16_lo(g), bf16_lo(u)), glu_fwd_seq(bf16_hi(g), bf16_hi(u)));
}

__device__ __forceinline__ void glu_bwd2(uint32_t g, uint32_t u, uint32_t d, uint32_t& dg,
                                         uint32_t& du) {
  float g0, u0, g1, u1;
  glu_bwd_seq(bf16_lo(g), bf16_lo(u), bf16_lo(d), g0, u0);
  glu_bwd_seq(bf16_hi(g), bf16_hi(u), bf16_hi(d), g1, u1);
  dg = bf16x2_neg_zero_to_pos(pack_bf16x2(g0, g1));
  du = bf16x2_neg_zero_to_pos(pack_bf16x2(u0, u1));
}

__device__ __forceinline__ int32_t valid_rows(int32_t rows, const int32_t* limit) {
  if (limit == nullptr) return rows;
  const int32_t v = *limit;
  return v < 0 ? 0 : (v > rows ? rows : v);
}

__global__ void __launch_bounds__(kGluThreads) glu_fwd_kernel(const uint4* __restrict__ fused,
                                                              uint4* __restrict__ out,
                                                              int32_t rows, int32_t f,
                                                              const int32_t* limit) {
  const int32_t L = valid_rows(rows, limit);
  const int vpr = f >> 3;  // 16-byte vectors per output row
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * kGluWarps;
  for (int r = blockIdx.x * kGluWarps + (threadIdx.x >> 5); r < L; r += stride) {
    const uint4* g_row = fused + static_cast<size_t>(r) * 2 * vpr;
    const uint4* u_row = g_row + vpr;
    uint4* o_row = out + static_cast<size_t>(r) * vpr;
    for (int v0 = lane; v0 < vpr; v0 += 32 * kFwdBatch) {
      uint4 g[kFwdBatch], u[kFwdBatch];
#pragma unroll
      for (int b = 0; b < kFwdBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr) {
          g[b] = ld_stream(g_row + v);
          u[b] = ld_stream(u_row + v);
        }
      }
#pragma unroll
      for (int b = 0; b < kFwdBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr)
          o_row[v] = make_uint4(glu2(g[b].x, u[b].x), glu2(g[b].y, u[b].y), glu2(g[b].z, u[b].z),
                                glu2(g[b].w, u[b].w));
      }
    }
  }
}

__global__ void __launch_bounds__(kGluThreads) glu_bwd_kernel(const uint4* __restrict__ fused,
                                                              const uint4* __restrict__ d_out,
                                                              uint4* __restrict__ d_fused,
                                                              int32_t rows, int32_t f,
                                                              const int32_t* limit) {
  const int32_t L = valid_rows(rows, limit);
  const int vpr = f >> 3;
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * kGluWarps;
  for (int r = blockIdx.x * kGluWarps + (threadIdx.x >> 5); r < L; r += stride) {
    const uint4* g_row = fused + static_cast<size_t>(r) * 2 * vpr;
    const uint4* u_row = g_row + vpr;
    const uint4* d_row = d_out + static_cast<size_t>(r) * vpr;
    uint4* dg_row = d_fused + static_cast<size_t>(r) * 2 * vpr;
    uint4* du_row = dg_row + vpr;
    for (int v0 = lane; v0 < vpr; v0 += 32 * kBwdBatch) {
      uint4 g[kBwdBatch], u[kBwdBatch], d[kBwdBatch];
#pragma unroll
      for (int b = 0; b < kBwdBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr) {
          g[b] = ld_stream(g_row + v);
          u[b] = ld_stream(u_row + v);
          d[b] = ld_stream(d_row + v);
        }
      }
#pragma unroll
      for (int b = 0; b < kBwdBatch; ++b) {
        const int v = v0 + 32 * b;
        if (v < vpr) {
          uint4 og, ou;
          glu_bwd2(g[b].x, u[b].x, d[b].x, og.x, ou.x);
          glu_bwd2(g[b].y, u[b].y, d[b].y, og.y, ou.y);
          glu_bwd2(g[b].z, u[b].z, d[b].z, og.z, ou.z);
          glu_bwd2(g[b].w, u[b].w, d[b].w, og.w, ou.w);
          dg_row[v] = og;
          du_row[v] = ou;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_glu_fwd(const void* fused, void* out, int32_t rows, int32_t f,
                           const int32_t* limit, int grid, cudaStream_t stream) {
  glu_fwd_kernel<<<grid, kGluThreads, 0, stream>>>(static_cast<const uint4*>(fused),
                                                   static_cast<uint4*>(out), rows, f, limit);
  return cudaGetLastError();
}

cudaError_t launch_glu_bwd(const void* fused, const void* d_out, void* d_fused, int32_t rows,
                           int32_t f, const int32_t* limit, int grid, cudaStream_t stream) {
  glu_bwd_kernel<<<grid, kGluThreads, 0, stream>>>(static_cast<const uint4*>(fused),
                                                   static_cast<const uint4*>(d_out),
                                                   static_cast<uint4*>(d_fused), rows, f, limit);
  return cudaGetLastError();
}

}  // namespace rd
