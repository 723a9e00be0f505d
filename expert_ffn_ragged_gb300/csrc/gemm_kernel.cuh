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
// How (one CTA per SM, 256 threads):
//   * every CTA reads group_sizes and *limit itself and builds the group
//     boundaries (exclusive prefix clamped to L) and the per-group tile
//     prefix in shared memory -- no workspace, no host round trip;
//   * tiles are handed out by static striding t = blockIdx.x + i * gridDim.x
//     over (group, m-tile, n-tile) with m fastest, so the CTAs working at one
//     time share each rhs column panel through L2;
//   * warp 0 (one lane) streams A/B blocks with TMA into a 4-stage ring of
//     128-byte-swizzled tiles; warp 1 issues tcgen05.mma 128x256x16 into one
//     of two TMEM accumulators; warps 2-5 drain the other accumulator with
//     tcgen05.ld, round to bf16 (or apply the GLU) and store with row masks;
//     warps 6-7 write the zero rows of the forward/dx outputs;
//   * the last m-tile of a group is loaded from row (end - 128) so no row at
//     or past the group end -- hence none at or past L -- is read; it stores
//     only the rows it owns.  dw uses the same shift on its row (K) blocks and
//     zeroes, in shared memory, the rows of a block that lie before the
//     group, so rows of other groups never enter the sum (NaN-safe);
//   * every wait is bounded; on expiry the CTA unwinds, drains its TMA and
//     MMA work, frees TMEM and reports RD_STATUS_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/rd.h"
#include "gemm_args.h"
#include "glu_math.cuh"
#include "ptx.cuh"

namespace rd {

struct alignas(16) GemmShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t L;
  int32_t total_tiles;
  int32_t zero_lo;  // forward/dx: rows [0, zero_lo) are zero
  int32_t zero_hi;  // forward/dx: rows [zero_hi, L) are zero
  int32_t bound[kMaxGroups + 1];       // group boundaries, clamped to L
  int32_t tile_start[kMaxGroups + 1];  // first tile of each local group
};

constexpr size_t kGemmSmemBytes =
    1024 + static_cast<size_t>(kStages) * (kStageBytesA + kStageBytesB) + sizeof(GemmShared);

// One unit of work as every role sees it.
struct Tile {
  int32_t j;         // local group
  int32_t m_idx;     // row tile (fwd/dx: within the group; dw: within the weight block)
  int32_t n_idx;     // column tile
  int32_t rs, re;    // rows of the group, clamped to L
  int32_t row_load;  // fwd/dx: first row the A tile is loaded from
  int32_t nkb;       // K blocks (0: the tile is all zeros)
};

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
template <int OP, bool GLU>
__device__ __forceinline__ void build_schedule(GemmShared& sh, const GemmArgs& a, int lane) {
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
    sh.bound[i] = static_cast<int32_t>(run < L ? run : L);
    const int s = a.group_sizes[i];
    run += s > 0 ? s : 0;
  }
  const long long total = __shfl_sync(0xFFFFFFFFu, run, 31);
  neg = __any_sync(0xFFFFFFFFu, neg);
  if (lane == 0) {
    sh.bound[G] = static_cast<int32_t>(total < L ? total : L);
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
  long long tsum = 0;
  for (int j = lo2; j < hi2; ++j) {
    if (OP == kOpDw) {
      tsum += static_cast<long long>(a.dw_m_tiles) * a.n_tiles;
    } else {
      const int cnt = sh.bound[a.group_offset + j + 1] - sh.bound[a.group_offset + j];
      tsum += static_cast<long long>((cnt + kBM - 1) / kBM) * a.n_tiles;
    }
  }
  long long trun = warp_exclusive_scan(tsum, lane);
  for (int j = lo2; j < hi2; ++j) {
    sh.tile_start[j] = static_cast<int32_t>(trun);
    if (OP == kOpDw) {
      trun += static_cast<long long>(a.dw_m_tiles) * a.n_tiles;
    } else {
      const int cnt = sh.bound[a.group_offset + j + 1] - sh.bound[a.group_offset + j];
      trun += static_cast<long long>((cnt + kBM - 1) / kBM) * a.n_tiles;
    }
  }
  const long long ttotal = __shfl_sync(0xFFFFFFFFu, trun, 31);
  if (lane == 0) {
    sh.tile_start[GL] = static_cast<int32_t>(ttotal);
    sh.total_tiles = static_cast<int32_t>(ttotal);
    sh.zero_lo = sh.bound[a.group_offset];
    sh.zero_hi = sh.bound[a.group_offset + GL];
  }
}

template <int OP>
__device__ __forceinline__ Tile decode_tile(const GemmShared& sh, const GemmArgs& a, int t) {
  Tile tl;
  if (OP == kOpDw) {
    const int per_group = a.dw_m_tiles * a.n_tiles;
    tl.j = t / per_group;
    const int u = t - tl.j * per_group;
    tl.m_idx = u % a.dw_m_tiles;
    tl.n_idx = u / a.dw_m_tiles;
    tl.rs = sh.bound[a.group_offset + tl.j];
    tl.re = sh.bound[a.group_offset + tl.j + 1];
    tl.row_load = 0;
    tl.nkb = (tl.re - tl.rs + kBK - 1) / kBK;
  } else {
    int lo = 0, hi = a.g_local;  // tile_start[lo] <= t < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sh.tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    tl.j = lo;
    const int u = t - sh.tile_start[lo];
    tl.rs = sh.bound[a.group_offset + lo];
    tl.re = sh.bound[a.group_offset + lo + 1];
    const int mt = (tl.re - tl.rs + kBM - 1) / kBM;
    tl.m_idx = u % mt;
    tl.n_idx = u / mt;
    const int first = tl.rs + tl.m_idx * kBM;
    tl.row_load = (tl.m_idx == mt - 1) ? tl.re - kBM : first;
    tl.nkb = (a.kc + kBK - 1) / kBK;
  }
  return tl;
}

// Store 32 consecutive bf16 (packed in 16 words) of one row, masked per 8 columns.
__device__ __forceinline__ void store_row32(__nv_bfloat16* row_ptr, int col, int n_out,
                                            const uint32_t (&p)[16]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    if (col + 8 * v + 8 <= n_out) {
      *reinterpret_cast<uint4*>(row_ptr + col + 8 * v) =
          make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
    }
  }
}

template <int OP, bool GLU>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageBytesA;
  GemmShared& sh = *reinterpret_cast<GemmShared*>(smem + kStages * (kStageBytesA + kStageBytesB));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&sh.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_addr(&sh.tfull[b]), 1);
      ptx::mbar_init(ptx::smem_addr(&sh.tempty[b]), 4);
    }
    ptx::mbar_init(ptx::smem_addr(&sh.drain), 1);
    sh.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && args.kc > 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&sh.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 2) build_schedule<OP, GLU>(sh, args, lane);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const int total = sh.total_tiles;
  const uint64_t tlimit = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pend_mask = 0, pend_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_tile<OP>(sh, args, t);
        for (int kb = 0; kb < tl.nkb; ++kb) {
          if (!ptx::mbar_wait_bounded(ptx::smem_addr(&sh.empty[stage]), phase ^ 1, abort_flag,
                                      tlimit)) {
            ok = false;
            break;
          }
          pend_mask &= ~(1u << stage);
          const uint32_t fb = ptx::smem_addr(&sh.full[stage]);
          ptx::mbar_arrive_expect_tx(fb, kStageBytesA + kStageBytesB);
          const uint32_t a_dst = ptx::smem_addr(sA + stage * kStageBytesA);
          const uint32_t b_dst = ptx::smem_addr(sB + stage * kStageBytesB);
          if (OP == kOpFwd) {
            ptx::tma_load_2d(a_dst, &tmap_a, fb, kb * kBK, tl.row_load);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int x = GLU ? ((c < 2 ? 0 : args.glu_f) + tl.n_idx * (kBN / 2) + (c & 1) * 64)
                                : (tl.n_idx * kBN + c * 64);
              ptx::tma_load_3d(b_dst + c * (kBK * 128), &tmap_b, fb, x, kb * kBK, tl.j);
            }
          } else if (OP == kOpDx) {
            ptx::tma_load_2d(a_dst, &tmap_a, fb, kb * kBK, tl.row_load);
            ptx::tma_load_3d(b_dst, &tmap_b, fb, kb * kBK, tl.n_idx * kBN, tl.j);
          } else {
            const int row0 = (kb == tl.nkb - 1) ? tl.re - kBK : tl.rs + kb * kBK;
#pragma unroll
            for (int c = 0; c < 2; ++c)
              ptx::tma_load_2d(a_dst + c * (kBK * 128), &tmap_a, fb, tl.m_idx * kBM + c * 64, row0);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              ptx::tma_load_2d(b_dst + c * (kBK * 128), &tmap_b, fb, tl.n_idx * kBN + c * 64, row0);
          }
          pend_mask |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA's shared memory goes away
        volatile int no_abort = 0;
        for (int s = 0; s < kStages; ++s)
          if (pend_mask & (1u << s))
            ptx::mbar_wait_bounded(ptx::smem_addr(&sh.full[s]), (pend_par >> s) & 1u, &no_abort,
                                   tlimit);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr bool a_mn = (OP == kOpDw);
    constexpr bool b_mn = (OP != kOpDx);
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, a_mn, b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode_tile<OP>(sh, args, t);
      if (tl.nkb == 0) continue;
      ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.tempty[acc]), acc_phase ^ 1, abort_flag,
                                  tlimit);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = sh.tmem_base + static_cast<uint32_t>(acc * kBN);
      for (int kb = 0; kb < tl.nkb; ++kb) {
        ok = ptx::mbar_wait_bounded(ptx::smem_addr(&sh.full[stage]), phase, abort_flag, tlimit);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        uint8_t* a_st = sA + stage * kStageBytesA;
        uint8_t* b_st = sB + stage * kStageBytesB;
        if (OP == kOpDw && kb == tl.nkb - 1) {
          // rows of the last block that precede this group's block start: zero them in
          // both operands so nothing from a neighbouring group (or a NaN) enters the sum
          const int rem = (tl.re - tl.rs) - (tl.nkb - 1) * kBK;
          const int zrows = kBK - rem;
          if (zrows > 0) {
            // each row is one 128-byte line per 64-wide chunk: 2 chunks of A, 4 of B
            const int units = zrows * 6 * 8;  // 16-byte units
            for (int u = lane; u < units; u += 32) {
              const int row = u / 48;
              const int rest = u - row * 48;
              const int chunk = rest >> 3;
              const int part = rest & 7;
              uint8_t* base = chunk < 2 ? a_st + chunk * (kBK * 128)
                                        : b_st + (chunk - 2) * (kBK * 128);
              *reinterpret_cast<uint4*>(base + row * 128 + part * 16) = make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t a_addr = ptx::smem_addr(a_st);
          const uint32_t b_addr = ptx::smem_addr(b_st);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = a_mn ? ptx::sw128_desc(a_addr + kk * 2048, kBK * 128, 1024)
                                        : ptx::sw128_desc(a_addr + kk * 32, 16, 1024);
            const uint64_t bdesc = b_mn ? ptx::sw128_desc(b_addr + kk * 2048, kBK * 128, 1024)
                                        : ptx::sw128_desc(b_addr + kk * 32, 16, 1024);
            ptx::tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::tc_commit(ptx::smem_addr(&sh.empty[stage]));
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) ptx::tc_commit(ptx::smem_addr(&sh.tfull[acc]));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (*abort_flag) {
      // wait until every MMA this thread issued has completed before TMEM is freed
      if (lane == 0) {
        volatile int no_abort = 0;
        ptx::tc_commit(ptx::smem_addr(&sh.drain));
        ptx::mbar_wait_bounded(ptx::smem_addr(&sh.drain), 0, &no_abort, tlimit);
      }
      __syncwarp();
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r_in_tile = q * 32 + lane;
    constexpr int tile_w = GLU ? kBN / 2 : kBN;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile<OP>(sh, args, t);
      // destination row of this thread and whether it owns it
      int row;
      bool valid;
      __nv_bfloat16* row_ptr;
      if (OP == kOpDw) {
        row = tl.m_idx * kBM + r_in_tile;
        valid = row < args.m_out;
        row_ptr = out + (static_cast<size_t>(tl.j) * args.m_out + row) * args.n_out;
      } else {
        row = tl.row_load + r_in_tile;
        valid = row >= tl.rs + tl.m_idx * kBM && row < tl.re;
        row_ptr = out + static_cast<size_t>(row) * args.n_out;
      }
      const int col0 = tl.n_idx * tile_w;
      if (tl.nkb == 0) {
        const uint32_t z[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        if (valid)
          for (int c = 0; c < tile_w / 32; ++c) store_row32(row_ptr, col0 + c * 32, args.n_out, z);
        continue;
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
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32], p[16];
          ptx::tmem_load_32cols(tbase + c * 32, g);
          ptx::tmem_load_32cols(tbase + kBN / 2 + c * 32, u);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(glu_fwd_f32(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                               glu_fwd_f32(__uint_as_float(g[2 * i + 1]),
                                           __uint_as_float(u[2 * i + 1])));
          if (valid) store_row32(row_ptr, col0 + c * 32, args.n_out, p);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32], p[16];
          ptx::tmem_load_32cols(tbase + c * 32, v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (valid) store_row32(row_ptr, col0 + c * 32, args.n_out, p);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sh.tempty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else if (OP != kOpDw) {
    // ------------------------------------------------------------ zero fill
    // rows [0, zero_lo) and [zero_hi, L): this CTA's contiguous share of them
    const long long zlo = sh.zero_lo;
    const long long zhi_n = sh.L - sh.zero_hi;
    const long long Z = zlo + zhi_n;
    const long long r0 = Z * blockIdx.x / gridDim.x;
    const long long r1 = Z * (blockIdx.x + 1) / gridDim.x;
    const int vpr = args.n_out / 8;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
    for (long long rc = r0 + (warp - 6); rc < r1; rc += 2) {
      const long long row = rc < zlo ? rc : sh.zero_hi + (rc - zlo);
      uint4* p = reinterpret_cast<uint4*>(out + row * args.n_out);
      for (int v = lane; v < vpr; v += 32) p[v] = make_uint4(0, 0, 0, 0);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(sh.tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && sh.abort_flag && args.status != nullptr)
    atomicOr(args.status, RD_STATUS_TIMEOUT);
}

template <int OP, bool GLU>
cudaError_t launch_gemm_impl(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                             const GemmArgs& args, int grid, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<OP, GLU>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kGemmSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  grouped_gemm_kernel<OP, GLU><<<grid, kThreads, kGemmSmemBytes, stream>>>(tmap_a, tmap_b, args);
  return cudaGetLastError();
}

}  // namespace rd
