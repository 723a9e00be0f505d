// api.cu -- the C ABI of librd (include/rd.h): argument checks, TMA tensor
// maps, launch shapes.  Every check that can be made on the host is made
// before any CUDA call, so bad arguments are rejected even without a GPU.
// Nothing here synchronises, allocates or copies device data to the host.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/rd.h"
#include "gemm_args.h"

namespace rd {
namespace {

constexpr uint64_t kTimeoutNs = 4000000000ull;  // default bound of any single wait in a kernel
constexpr int32_t kBandRows = 6144;              // default rows per band of the fwd/dx tile order

// Process-wide tuning overrides (rd_set_tuning); 0 = the default.
std::atomic<int32_t> g_variant{RD_VARIANT_AUTO};
std::atomic<int32_t> g_band_rows{0};
std::atomic<uint64_t> g_timeout_ns{0};

uint64_t wait_timeout_ns() {
  const uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
  return t == 0 ? kTimeoutNs : t;
}
constexpr int64_t kMaxDim = 0x7FFFFFFF;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// SM count of the current device, and whether it is an sm_103 part
rd_status current_device(int* sms) {
  static std::mutex mu;
  static int cached_sms[64];
  static int cached_state[64];  // 0 unknown, 1 supported, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RD_ERR_CUDA;
  if (dev < 0 || dev >= 64) return RD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (cached_state[dev] == 0) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return RD_ERR_CUDA;
    cached_sms[dev] = count;
    cached_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  *sms = cached_sms[dev];
  return cached_state[dev] == 1 ? RD_OK : RD_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first.
// Encoding costs about a microsecond of host time, a large share of a small
// call, so each thread keeps the last few maps it encoded (a map is a pure
// function of these arguments).
struct MapKey {
  const void* base;
  int rank;
  uint64_t dims[5];
  uint64_t strides[4];
  uint32_t box[5];
};

rd_status encode(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box) {
  constexpr int kCache = 16;
  struct Entry {
    MapKey key;
    CUtensorMap map;
    bool valid;
  };
  thread_local Entry cache[kCache];
  thread_local int next_slot = 0;
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) key.strides[i] = strides_bytes[i];
  for (int e = 0; e < kCache; ++e) {
    if (cache[e].valid && std::memcmp(&cache[e].key, &key, sizeof(key)) == 0) {
      *map = cache[e].map;
      return RD_OK;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return RD_ERR_CUDA;
  cuuint64_t gdim[5], gstride[4];
  cuuint32_t gbox[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    gbox[i] = box[i];
    estride[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gstride[i] = strides_bytes[i];
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim, gstride,
         gbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return RD_ERR_UNSUPPORTED;
  Entry& slot = cache[next_slot];
  next_slot = (next_slot + 1) % kCache;
  slot.key = key;
  slot.map = *map;
  slot.valid = true;
  return RD_OK;
}

// checks shared by the three grouped calls
rd_status check_groups(int64_t m, int64_t k, int64_t n, const int32_t* group_sizes,
                       int32_t g_total, int32_t group_offset, int32_t g_local,
                       const int32_t* limit, const int32_t* status) {
  if (m < 0 || k < 0 || n < 0) return RD_ERR_INVALID_ARG;
  if (group_sizes == nullptr) return RD_ERR_INVALID_ARG;
  if (g_total < 1 || g_local < 1 || group_offset < 0 ||
      static_cast<int64_t>(group_offset) + g_local > g_total)
    return RD_ERR_INVALID_ARG;
  if (g_total > RD_MAX_GROUPS) return RD_ERR_UNSUPPORTED;
  if (m > kMaxDim || k > kMaxDim || n > kMaxDim) return RD_ERR_UNSUPPORTED;
  if (k % 8 != 0 || n % 8 != 0) return RD_ERR_UNSUPPORTED;
  const uintptr_t a4 = 3u;
  if ((reinterpret_cast<uintptr_t>(group_sizes) & a4) || (reinterpret_cast<uintptr_t>(limit) & a4) ||
      (reinterpret_cast<uintptr_t>(status) & a4))
    return RD_ERR_UNSUPPORTED;
  return RD_OK;
}

// the output must not overlap any input (or the control words)
bool out_aliases(const void* out, uint64_t out_bytes, const void* in0, uint64_t b0,
                 const void* in1, uint64_t b1, const void* gs, uint64_t bgs, const void* limit,
                 const void* status) {
  return overlap(out, out_bytes, in0, b0) || overlap(out, out_bytes, in1, b1) ||
         overlap(out, out_bytes, gs, bgs) || overlap(out, out_bytes, limit, 4) ||
         overlap(out, out_bytes, status, 4);
}

int grid_for(int sms, int64_t tiles_upper_bound) {
  int64_t g = tiles_upper_bound < 1 ? 1 : tiles_upper_bound;
  return static_cast<int>(g < sms ? g : sms);
}

// Forward and dx run either on single CTAs (128x256 tiles) or on CTA pairs
// (256x256 tiles, cta_group::2).  Pairs halve the operand bytes each SM pulls
// per MMA and win when groups are large; with small groups (decode-shaped
// calls, a few rows per expert) the 256-row tile mostly computes padding and
// single CTAs stream the weights faster.  The choice uses host-known shapes
// only: pairs when the buffer holds at least 512 rows per group on average.
// rd_set_tuning can force either variant.
bool use_pair(int sms, int64_t m, int32_t g_total) {
  if (sms < 2) return false;
  const int32_t v = g_variant.load(std::memory_order_relaxed);
  if (v == RD_VARIANT_SINGLE) return false;
  if (v == RD_VARIANT_PAIR) return true;
  return m >= 512 * static_cast<int64_t>(g_total);
}

// m-tiles per band of the forward / dx tile order: the band's lhs rows stay in
// L2 while the band sweeps every output column block.
int32_t band_tiles(bool pair) {
  const int32_t r = g_band_rows.load(std::memory_order_relaxed);
  const int64_t rows = r > 0 ? r : kBandRows;
  const int64_t tile = pair ? 2 * kBM : kBM;
  const int64_t t = rows / tile;
  return static_cast<int32_t>(t < 1 ? 1 : t);
}

int pair_grid(int sms, int64_t pair_tiles_upper_bound) {
  return 2 * grid_for(sms / 2, pair_tiles_upper_bound);
}

}  // namespace
}  // namespace rd

using namespace rd;

extern "C" rd_status rd_ragged_dot(const void* lhs, const void* rhs, void* out, int64_t m,
                                   int64_t k, int64_t n, const int32_t* group_sizes,
                                   int32_t g_total, int32_t group_offset, int32_t g_local,
                                   const int32_t* limit, rd_epilogue epi, int32_t* status,
                                   rd_stream_t stream) {
  const bool glu = epi == RD_EPI_SILU_GLU;
  if (epi != RD_EPI_NONE && !glu) return RD_ERR_INVALID_ARG;
  rd_status st = check_groups(m, k, n, group_sizes, g_total, group_offset, g_local, limit, status);
  if (st != RD_OK) return st;
  if (glu && n % 16 != 0) return n % 2 ? RD_ERR_INVALID_ARG : RD_ERR_UNSUPPORTED;
  const int64_t n_out = glu ? n / 2 : n;
  if ((m > 0 && k > 0 && lhs == nullptr) || (k > 0 && n > 0 && rhs == nullptr) ||
      (m > 0 && n_out > 0 && out == nullptr))
    return RD_ERR_INVALID_ARG;
  if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out)) return RD_ERR_UNSUPPORTED;
  const uint64_t out_bytes = static_cast<uint64_t>(m) * n_out * 2;
  if (out_aliases(out, out_bytes, lhs, static_cast<uint64_t>(m) * k * 2, rhs,
                  static_cast<uint64_t>(g_local) * k * n * 2, group_sizes,
                  static_cast<uint64_t>(g_total) * 4, limit, status))
    return RD_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (m == 0 || n_out == 0) return RD_OK;

  CUtensorMap ta = {}, tb = {};
  if (k > 0) {
    const uint64_t da[2] = {static_cast<uint64_t>(k), static_cast<uint64_t>(m)};
    const uint64_t sa[1] = {static_cast<uint64_t>(k) * 2};
    const uint32_t ba[2] = {64, kBM};
    if ((st = encode(&ta, lhs, 2, da, sa, ba)) != RD_OK) return st;
    const uint64_t db[3] = {static_cast<uint64_t>(n), static_cast<uint64_t>(k),
                            static_cast<uint64_t>(g_local)};
    const uint64_t sb[2] = {static_cast<uint64_t>(n) * 2, static_cast<uint64_t>(k) * n * 2};
    const uint32_t bb[3] = {64, kBK, 1};
    if ((st = encode(&tb, rhs, 3, db, sb, bb)) != RD_OK) return st;
  }
  GemmArgs a = {};
  a.group_sizes = group_sizes;
  a.limit = limit;
  a.status = status;
  a.out = out;
  a.m = static_cast<int32_t>(m);
  a.kc = static_cast<int32_t>(k);
  a.n_out = static_cast<int32_t>(n_out);
  a.m_out = 0;
  a.g_total = g_total;
  a.group_offset = group_offset;
  a.g_local = g_local;
  a.glu_f = static_cast<int32_t>(n_out);
  a.ldo = n_out;
  a.zero_cols = static_cast<int32_t>(n_out);
  const int tile_w = glu ? kBN / 2 : kBN;
  a.n_tiles = static_cast<int32_t>((n_out + tile_w - 1) / tile_w);
  a.dw_m_tiles = 0;
  a.timeout_ns = wait_timeout_ns();
  const bool pair = use_pair(sms, m, g_total);
  a.band_tiles = band_tiles(pair);
  const int grid = pair ? pair_grid(sms, ((m + 2 * kBM - 1) / (2 * kBM) + g_local) * a.n_tiles)
                        : grid_for(sms, ((m + kBM - 1) / kBM + g_local) * a.n_tiles);
  return launch_gemm_fwd(glu, pair, ta, tb, a, grid, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}

namespace {
// rd_ragged_dot_trans_rhs, optionally followed (in the epilogue) by the SiLU-GLU
// backward against the saved fused buffer: out = dx [m, k], or [d_gate | d_up]
// [m, 2k] when fused != nullptr.
rd_status trans_rhs_impl(const void* lhs, const void* rhs, const void* fused, void* out, int64_t m,
                         int64_t k, int64_t n, const int32_t* group_sizes, int32_t g_total,
                         int32_t group_offset, int32_t g_local, const int32_t* limit,
                         int32_t* status, rd_stream_t stream) {
  rd_status st = check_groups(m, k, n, group_sizes, g_total, group_offset, g_local, limit, status);
  if (st != RD_OK) return st;
  const bool glu_bwd = fused != nullptr;
  const int64_t out_w = glu_bwd ? 2 * k : k;
  if ((m > 0 && n > 0 && lhs == nullptr) || (k > 0 && n > 0 && rhs == nullptr) ||
      (m > 0 && k > 0 && out == nullptr))
    return RD_ERR_INVALID_ARG;
  if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || !aligned16(fused))
    return RD_ERR_UNSUPPORTED;
  const uint64_t ob = static_cast<uint64_t>(m) * out_w * 2;
  if (out_aliases(out, ob, lhs, static_cast<uint64_t>(m) * n * 2, rhs,
                  static_cast<uint64_t>(g_local) * k * n * 2, group_sizes,
                  static_cast<uint64_t>(g_total) * 4, limit, status) ||
      overlap(out, ob, fused, static_cast<uint64_t>(m) * 2 * k * 2))
    return RD_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (m == 0 || k == 0) return RD_OK;

  const bool pair = use_pair(sms, m, g_total);
  CUtensorMap ta = {}, tb = {};
  if (n > 0) {
    const uint64_t da[2] = {static_cast<uint64_t>(n), static_cast<uint64_t>(m)};
    const uint64_t sa[1] = {static_cast<uint64_t>(n) * 2};
    const uint32_t ba[2] = {64, kBM};
    if ((st = encode(&ta, lhs, 2, da, sa, ba)) != RD_OK) return st;
    const uint64_t db[3] = {static_cast<uint64_t>(n), static_cast<uint64_t>(k),
                            static_cast<uint64_t>(g_local)};
    const uint64_t sb[2] = {static_cast<uint64_t>(n) * 2, static_cast<uint64_t>(k) * n * 2};
    // each CTA of a pair holds half of the 256 output columns
    const uint32_t bb[3] = {64, static_cast<uint32_t>(pair ? kBN / 2 : kBN), 1};
    if ((st = encode(&tb, rhs, 3, db, sb, bb)) != RD_OK) return st;
  }
  GemmArgs a = {};
  a.group_sizes = group_sizes;
  a.limit = limit;
  a.status = status;
  a.out = out;
  a.aux = fused;
  a.ldo = out_w;
  a.zero_cols = static_cast<int32_t>(out_w);
  a.m = static_cast<int32_t>(m);
  a.kc = static_cast<int32_t>(n);
  a.n_out = static_cast<int32_t>(k);
  a.g_total = g_total;
  a.group_offset = group_offset;
  a.g_local = g_local;
  a.n_tiles = static_cast<int32_t>((k + kBN - 1) / kBN);
  a.band_tiles = band_tiles(pair);
  a.timeout_ns = wait_timeout_ns();
  const int grid = pair ? pair_grid(sms, ((m + 2 * kBM - 1) / (2 * kBM) + g_local) * a.n_tiles)
                        : grid_for(sms, ((m + kBM - 1) / kBM + g_local) * a.n_tiles);
  return launch_gemm_dx(pair, glu_bwd, ta, tb, a, grid, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}
}  // namespace

extern "C" rd_status rd_ragged_dot_trans_rhs(const void* lhs, const void* rhs, void* out,
                                             int64_t m, int64_t k, int64_t n,
                                             const int32_t* group_sizes, int32_t g_total,
                                             int32_t group_offset, int32_t g_local,
                                             const int32_t* limit, int32_t* status,
                                             rd_stream_t stream) {
  return trans_rhs_impl(lhs, rhs, nullptr, out, m, k, n, group_sizes, g_total, group_offset,
                        g_local, limit, status, stream);
}

extern "C" rd_status rd_ragged_dot_trans_rhs_glu_bwd(const void* d_out, const void* rhs,
                                                     const void* fused, void* d_fused, int64_t m,
                                                     int64_t f, int64_t n,
                                                     const int32_t* group_sizes, int32_t g_total,
                                                     int32_t group_offset, int32_t g_local,
                                                     const int32_t* limit, int32_t* status,
                                                     rd_stream_t stream) {
  if (m > 0 && f > 0 && fused == nullptr) return RD_ERR_INVALID_ARG;
  // a null fused buffer (only possible for an empty problem) still selects the GLU form
  static const int32_t dummy[4] = {0, 0, 0, 0};
  return trans_rhs_impl(d_out, rhs, fused != nullptr ? fused : static_cast<const void*>(dummy),
                        d_fused, m, f, n, group_sizes, g_total, group_offset, g_local, limit,
                        status, stream);
}

namespace {
// trans_ragged_dot with a bf16 (epi = kEpiNone) or f32 (kEpiF32, kEpiF32Acc) output
rd_status trans_ragged_impl(const void* x, const void* y, void* out, int64_t m, int64_t k,
                            int64_t n, const int32_t* group_sizes, int32_t g_total,
                            int32_t group_offset, int32_t g_local, const int32_t* limit,
                            int epi, void* workspace, size_t workspace_bytes, int32_t* status,
                            rd_stream_t stream) {
  const uint64_t out_elem = epi == kEpiNone ? 2 : 4;
  rd_status st = check_groups(m, k, n, group_sizes, g_total, group_offset, g_local, limit, status);
  if (st != RD_OK) return st;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 127u))
    return RD_ERR_UNSUPPORTED;
  if ((m > 0 && k > 0 && x == nullptr) || (m > 0 && n > 0 && y == nullptr) ||
      (k > 0 && n > 0 && out == nullptr))
    return RD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(out)) return RD_ERR_UNSUPPORTED;
  if (out_aliases(out, static_cast<uint64_t>(g_local) * k * n * out_elem, x,
                  static_cast<uint64_t>(m) * k * 2, y, static_cast<uint64_t>(m) * n * 2,
                  group_sizes, static_cast<uint64_t>(g_total) * 4, limit, status))
    return RD_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  // the workspace holds the per-group maps of every CTA; it must not overlap
  // anything the call reads or writes
  const uint64_t ws_need = static_cast<uint64_t>(sms) * kMapBytesPerCta;
  if (workspace != nullptr &&
      (workspace_bytes < ws_need ||
       out_aliases(workspace, workspace_bytes, x, static_cast<uint64_t>(m) * k * 2, y,
                   static_cast<uint64_t>(m) * n * 2, group_sizes,
                   static_cast<uint64_t>(g_total) * 4, limit, status) ||
       overlap(workspace, workspace_bytes, out, static_cast<uint64_t>(g_local) * k * n * out_elem)))
    return RD_ERR_INVALID_ARG;
  if (k == 0 || n == 0) return RD_OK;

  const bool pair = use_pair(sms, m, g_total);
  // Both operands are MN-major (the token rows are the contraction).  When a
  // width is a multiple of 64 its map is 3-D, (64 columns, rows, 64-column
  // chunks), so that one box brings all the chunks of a stage (the producer
  // issues half as many copies); otherwise one 2-D box per 64 columns, whose
  // zero fill covers the columns past the width.
  const bool a_chunked = k % 64 == 0, b_chunked = n % 64 == 0;
  CUtensorMap ta = {}, tb = {};
  if (m > 0) {
    if (a_chunked) {
      const uint64_t da[3] = {64, static_cast<uint64_t>(m), static_cast<uint64_t>(k / 64)};
      const uint64_t sa[2] = {static_cast<uint64_t>(k) * 2, 128};
      const uint32_t ba[3] = {64, kBK, kBM / 64};
      if ((st = encode(&ta, x, 3, da, sa, ba)) != RD_OK) return st;
    } else {
      const uint64_t da[2] = {static_cast<uint64_t>(k), static_cast<uint64_t>(m)};
      const uint64_t sa[1] = {static_cast<uint64_t>(k) * 2};
      const uint32_t ba[2] = {64, kBK};
      if ((st = encode(&ta, x, 2, da, sa, ba)) != RD_OK) return st;
    }
    if (b_chunked) {
      const uint64_t db[3] = {64, static_cast<uint64_t>(m), static_cast<uint64_t>(n / 64)};
      const uint64_t sb[2] = {static_cast<uint64_t>(n) * 2, 128};
      const uint32_t bb[3] = {64, kBK, static_cast<uint32_t>((pair ? kBN / 2 : kBN) / 64)};
      if ((st = encode(&tb, y, 3, db, sb, bb)) != RD_OK) return st;
    } else {
      const uint64_t db[2] = {static_cast<uint64_t>(n), static_cast<uint64_t>(m)};
      const uint64_t sb[1] = {static_cast<uint64_t>(n) * 2};
      const uint32_t bb[2] = {64, kBK};
      if ((st = encode(&tb, y, 2, db, sb, bb)) != RD_OK) return st;
    }
  }
  const int tile_rows = pair ? 2 * kBM : kBM;  // rows of dw[j] (the k axis) per tile
  GemmArgs a = {};
  a.a_chunked = a_chunked ? 1 : 0;
  a.b_chunked = b_chunked ? 1 : 0;
  a.group_sizes = group_sizes;
  a.limit = limit;
  a.status = status;
  a.out = out;
  a.m = static_cast<int32_t>(m);
  a.kc = static_cast<int32_t>(m);
  a.n_out = static_cast<int32_t>(n);
  a.m_out = static_cast<int32_t>(k);
  a.ldo = n;
  a.zero_cols = static_cast<int32_t>(n);
  a.g_total = g_total;
  a.group_offset = group_offset;
  a.g_local = g_local;
  a.n_tiles = static_cast<int32_t>((n + kBN - 1) / kBN);
  a.dw_m_tiles = static_cast<int32_t>((k + tile_rows - 1) / tile_rows);
  // with a workspace each CTA rebases the maps to each group it works on (rows
  // outside the group then arrive as zeros); without one the edge rows of each
  // group's first block are zeroed in shared memory
  a.group_maps = workspace != nullptr ? 1 : 0;
  a.x_base = x;
  a.y_base = y;
  a.x_row_bytes = k * 2;
  a.y_row_bytes = n * 2;
  a.maps = static_cast<CUtensorMap*>(workspace);
  a.timeout_ns = wait_timeout_ns();
  const int64_t tiles = static_cast<int64_t>(g_local) * a.dw_m_tiles * a.n_tiles;
  if (tiles > kMaxDim) return RD_ERR_UNSUPPORTED;
  const int grid = pair ? pair_grid(sms, tiles) : grid_for(sms, tiles);
  return launch_gemm_dw(pair, epi, ta, tb, a, grid, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}
}  // namespace

extern "C" rd_status rd_trans_ragged_dot(const void* x, const void* y, void* out, int64_t m,
                                         int64_t k, int64_t n, const int32_t* group_sizes,
                                         int32_t g_total, int32_t group_offset, int32_t g_local,
                                         const int32_t* limit, void* workspace,
                                         size_t workspace_bytes, int32_t* status,
                                         rd_stream_t stream) {
  return trans_ragged_impl(x, y, out, m, k, n, group_sizes, g_total, group_offset, g_local, limit,
                           kEpiNone, workspace, workspace_bytes, status, stream);
}

extern "C" rd_status rd_trans_ragged_dot_workspace_size(size_t* bytes) {
  if (bytes == nullptr) return RD_ERR_INVALID_ARG;
  int sms = 0;
  const rd_status st = current_device(&sms);
  if (st != RD_OK) return st;
  *bytes = static_cast<size_t>(sms) * kMapBytesPerCta;
  return RD_OK;
}

extern "C" rd_status rd_trans_ragged_dot_f32(const void* x, const void* y, float* out, int64_t m,
                                             int64_t k, int64_t n, const int32_t* group_sizes,
                                             int32_t g_total, int32_t group_offset,
                                             int32_t g_local, const int32_t* limit,
                                             int32_t accumulate, void* workspace,
                                             size_t workspace_bytes, int32_t* status,
                                             rd_stream_t stream) {
  if (accumulate != 0 && accumulate != 1) return RD_ERR_INVALID_ARG;
  return trans_ragged_impl(x, y, out, m, k, n, group_sizes, g_total, group_offset, g_local, limit,
                           accumulate ? kEpiF32Acc : kEpiF32, workspace, workspace_bytes, status,
                           stream);
}

namespace {
rd_status check_glu(const void* a, const void* b, const void* out, int64_t rows, int64_t f,
                    const int32_t* limit) {
  if (rows < 0 || f < 0) return RD_ERR_INVALID_ARG;
  if (rows > kMaxDim || f > kMaxDim / 2) return RD_ERR_UNSUPPORTED;
  if (f % 8 != 0) return RD_ERR_UNSUPPORTED;
  if (rows > 0 && f > 0 && (a == nullptr || b == nullptr || out == nullptr))
    return RD_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(limit) & 3u))
    return RD_ERR_UNSUPPORTED;
  return RD_OK;
}
}  // namespace

extern "C" rd_status rd_glu_fwd(const void* fused, void* out, int64_t rows, int64_t f,
                                const int32_t* limit, rd_stream_t stream) {
  rd_status st = check_glu(fused, fused, out, rows, f, limit);
  if (st != RD_OK) return st;
  if (overlap(out, static_cast<uint64_t>(rows) * f * 2, fused,
              static_cast<uint64_t>(rows) * f * 4) ||
      overlap(out, static_cast<uint64_t>(rows) * f * 2, limit, 4))
    return RD_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (rows == 0 || f == 0) return RD_OK;
  const int grid = grid_for(sms * 8, (rows + 7) / 8);
  return launch_glu_fwd(fused, out, static_cast<int32_t>(rows), static_cast<int32_t>(f), limit,
                        grid, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}

extern "C" rd_status rd_glu_bwd(const void* fused, const void* d_out, void* d_fused, int64_t rows,
                                int64_t f, const int32_t* limit, rd_stream_t stream) {
  rd_status st = check_glu(fused, d_out, d_fused, rows, f, limit);
  if (st != RD_OK) return st;
  const uint64_t ob = static_cast<uint64_t>(rows) * f * 4;
  if (overlap(d_fused, ob, fused, ob) ||
      overlap(d_fused, ob, d_out, static_cast<uint64_t>(rows) * f * 2) ||
      overlap(d_fused, ob, limit, 4))
    return RD_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (rows == 0 || f == 0) return RD_OK;
  const int grid = grid_for(sms * 8, (rows + 7) / 8);
  return launch_glu_bwd(fused, d_out, d_fused, static_cast<int32_t>(rows),
                        static_cast<int32_t>(f), limit, grid,
                        reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}

extern "C" rd_status rd_unsort_bwd_rows(const void* g, const void* y, const float* w, void* grad,
                                        float* dot, int64_t rows, int64_t hidden,
                                        const int32_t* limit, rd_stream_t stream) {
  if (rows < 0 || hidden < 0) return RD_ERR_INVALID_ARG;
  if (rows > kMaxDim || hidden > kMaxDim) return RD_ERR_UNSUPPORTED;
  if (hidden % 8 != 0) return RD_ERR_UNSUPPORTED;
  if (rows > 0 && (w == nullptr || dot == nullptr)) return RD_ERR_INVALID_ARG;
  if (rows > 0 && hidden > 0 && (g == nullptr || y == nullptr || grad == nullptr))
    return RD_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(y) || !aligned16(grad) ||
      (reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(dot) & 3u) ||
      (reinterpret_cast<uintptr_t>(limit) & 3u))
    return RD_ERR_UNSUPPORTED;
  const uint64_t mb = static_cast<uint64_t>(rows) * hidden * 2, rb = static_cast<uint64_t>(rows) * 4;
  if (overlap(grad, mb, g, mb) || overlap(grad, mb, y, mb) || overlap(grad, mb, w, rb) ||
      overlap(grad, mb, dot, rb) || overlap(grad, mb, limit, 4) || overlap(dot, rb, g, mb) ||
      overlap(dot, rb, y, mb) || overlap(dot, rb, w, rb) || overlap(dot, rb, limit, 4))
    return RD_ERR_INVALID_ARG;
  rd_status st;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (rows == 0) return RD_OK;
  const int grid = grid_for(sms * 8, (rows + 7) / 8);
  return launch_unsort_bwd_rows(g, y, w, grad, dot, static_cast<int32_t>(rows),
                                static_cast<int32_t>(hidden), limit, grid,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RD_OK
             : RD_ERR_CUDA;
}

// ------------------------------------------------ dw without any allocation
// Some callers cannot allocate device memory at the point where they run the
// weight gradient: code inside an allocator's own callbacks, a runtime that
// owns every allocation and hands out no scratch, or a process that must not
// grow its footprint once set up.  For them rd_trans_ragged_dot_no_alloc runs
// the per-group-descriptor form of the dw kernel with its scratch in this
// file-scope array, which every GPU that loads the library holds until exit.
// It covers devices of up to kNoAllocMaxSms SMs (2 KB of descriptors per SM).
constexpr int kNoAllocMaxSms = 256;
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(kNoAllocMaxSms) * kMapBytesPerCta;
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

namespace {
// The array's device address on the current device.  In host code the array's
// name only stands in for the symbol: its address must come from the runtime,
// once per device, with that device current.
rd_status no_alloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RD_ERR_CUDA;
  if (dev < 0 || dev >= 64) return RD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || p == nullptr)
      return RD_ERR_CUDA;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return RD_OK;
}
}  // namespace

extern "C" rd_status rd_trans_ragged_dot_no_alloc(const void* x, const void* y, void* out, int64_t m,
                                                  int64_t k, int64_t n, const int32_t* group_sizes,
                                                  int32_t g_total, int32_t group_offset,
                                                  int32_t g_local, const int32_t* limit,
                                                  int32_t* status, rd_stream_t stream) {
  // the argument checks every dw call makes, before any CUDA call
  rd_status st = check_groups(m, k, n, group_sizes, g_total, group_offset, g_local, limit, status);
  if (st != RD_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != RD_OK) return st;
  if (sms > kNoAllocMaxSms) return RD_ERR_UNSUPPORTED;  // more CTAs than the array has room for
  void* scratch = nullptr;
  if ((st = no_alloc_scratch(&scratch)) != RD_OK) return st;
  return trans_ragged_impl(x, y, out, m, k, n, group_sizes, g_total, group_offset, g_local, limit,
                           kEpiNone, scratch, kNoAllocScratchBytes, status, stream);
}

extern "C" rd_status rd_set_tuning(const rd_tuning* t) {
  if (t == nullptr) {
    g_variant.store(RD_VARIANT_AUTO);
    g_band_rows.store(0);
    g_timeout_ns.store(0);
    return RD_OK;
  }
  if (t->gemm_variant < RD_VARIANT_AUTO || t->gemm_variant > RD_VARIANT_PAIR ||
      t->band_rows < 0 || t->reserved[0] != 0 || t->reserved[1] != 0)
    return RD_ERR_INVALID_ARG;
  g_variant.store(t->gemm_variant);
  g_band_rows.store(t->band_rows);
  g_timeout_ns.store(t->wait_timeout_ns);
  return RD_OK;
}

extern "C" rd_status rd_get_tuning(rd_tuning* t) {
  if (t == nullptr) return RD_ERR_INVALID_ARG;
  t->gemm_variant = g_variant.load();
  t->band_rows = g_band_rows.load();
  t->wait_timeout_ns = g_timeout_ns.load();
  t->reserved[0] = t->reserved[1] = 0;
  return RD_OK;
}

extern "C" const char* rd_status_string(rd_status s) {
  switch (s) {
    case RD_OK: return "RD_OK";
    case RD_ERR_INVALID_ARG: return "RD_ERR_INVALID_ARG: invalid argument";
    case RD_ERR_UNSUPPORTED: return "RD_ERR_UNSUPPORTED: unsupported shape, alignment or device";
    case RD_ERR_CUDA: return "RD_ERR_CUDA: CUDA runtime error";
  }
  return "unknown rd_status";
}
