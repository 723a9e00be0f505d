/*
 * rd.h -- C ABI of librd: the MoE ragged_dot (grouped GEMM) hot path on
 * NVIDIA GB300 (sm_103a).
 *
 * Every entry point takes plain device pointers and sizes, enqueues work on
 * the caller's CUDA stream and returns at once.  The library never
 * synchronises, never copies device data to the host and allocates nothing
 * (the dw calls can use a small workspace the caller provides); group_sizes
 * and limit stay on the device and are read by the kernels themselves.  A call can therefore be captured in a CUDA graph,
 * and replays follow device-side changes to group_sizes and limit.  The
 * first call of each entry point in a process sets a kernel attribute
 * (dynamic shared memory size); make it before a stream capture begins.
 *
 * Layout: every matrix is row-major and contiguous, bf16 unless stated.
 * Ownership: the caller owns every buffer; the library keeps no pointer
 * after the call returns (the work it enqueued still reads and writes the
 * buffers until it completes on the stream).
 *
 * Group semantics (all grouped calls):
 *   L      = min(max(*limit, 0), m), or m when limit is NULL.
 *   s[i]   = min(sum_{j<i} max(group_sizes[j], 0), L), i = 0..g_total.
 *   Group i owns rows [s[i], s[i+1]).  Local group j (0 <= j < g_local) is
 *   global group group_offset + j and uses rhs / weight block j.
 *   Rows in [0, L) outside the local groups are written as +0; rows >= L of
 *   every output are never written and rows >= L of every input are never
 *   read.
 *
 * Errors: invalid arguments are rejected before anything is enqueued
 * (RD_ERR_INVALID_ARG / RD_ERR_UNSUPPORTED); a failed launch returns
 * RD_ERR_CUDA.  Bad data found on the device (a negative group size, sizes
 * summing past m, a bounded wait that ran out) never traps: the kernel
 * clamps and, when `status` is not NULL, ORs an RD_STATUS_* bit into
 * *status.  The library never clears *status.
 *
 * Bounded waits: every wait inside the grouped-GEMM kernels gives up after
 * 4 s (rd_set_tuning can change the bound).  A kernel that gives up finishes
 * its copies and MMAs in flight, frees its tensor memory, returns, and sets
 * RD_STATUS_TIMEOUT; its outputs are then incomplete but the CUDA context
 * stays usable.  Pass a status word to see this: without one a timed-out
 * call is indistinguishable from a completed one.  An accumulating call
 * (rd_trans_ragged_dot_f32 with accumulate = 1) that timed out has added
 * some tiles and not others, so its output buffer is unusable (a retry
 * would add those tiles twice).
 *
 * The library reads no environment variable.
 */
#ifndef RD_H_
#define RD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* rd_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  RD_OK = 0,
  RD_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad group range, aliasing */
  RD_ERR_UNSUPPORTED = 2, /* width not a multiple of 8, misaligned pointer, too many groups, not sm_103 */
  RD_ERR_CUDA = 3         /* the CUDA runtime reported an error at launch */
} rd_status;

typedef enum {
  RD_EPI_NONE = 0,    /* store the f32 accumulator rounded to bf16 */
  RD_EPI_SILU_GLU = 1 /* out[:, c] = bf16(silu(acc[:, c]) * acc[:, F + c]), F = n / 2 */
} rd_epilogue;

/* device status bits, ORed into *status */
#define RD_STATUS_NEG_SIZE 1 /* a group size < 0 was taken as 0 */
#define RD_STATUS_OVERFLOW 2 /* the group sizes sum past m; boundaries clamped */
#define RD_STATUS_TIMEOUT 4  /* a bounded wait inside a kernel ran out; outputs incomplete */

/* largest g_total accepted by the grouped calls */
#define RD_MAX_GROUPS 1024

/*
 * rd_ragged_dot -- grouped forward.
 *   out[i, :] = lhs[i, :] @ rhs[j, :, :] for every row i of local group j.
 * Defined by SkyRL PR #867 "Integrate ragged_dot pallas kernel with
 * group_offset support" (the suggested fast_ragged_dot body: group
 * boundaries from a cumulative sum with an initial zero, only the local
 * groups computed, rows outside them zeroed) and MaxText PR #5760 "MoE wo
 * FSDP sharding and valid-rows-only MoE kernels" (commit message: only rows
 * [0, limit) of the packed buffer are valid; the SiLU-GLU over the fused
 * [gate | up] buffer, computed in f32 and rounded only at the output).
 *
 *   lhs          [m, k] bf16, device
 *   rhs          [g_local, k, n] bf16, device
 *   out          [m, n] bf16 (epi = NONE) or [m, n/2] (epi = SILU_GLU), device
 *   group_sizes  [g_total] int32, device
 *   group_offset first local group (host int), 0 <= group_offset,
 *                group_offset + g_local <= g_total <= RD_MAX_GROUPS
 *   limit        device int32 scalar or NULL
 *   epi          RD_EPI_NONE or RD_EPI_SILU_GLU (gate = columns [0, n/2) of
 *                the product, up = columns [n/2, n))
 *   status       device int32 or NULL
 * Accumulation is f32; the bf16 store rounds to nearest even.
 * Requires k % 8 == 0, n % 8 == 0 (n/2 % 8 == 0 with the GLU) and 16-byte
 * aligned pointers; out must not overlap lhs, rhs or group_sizes.
 */
rd_status rd_ragged_dot(const void* lhs, const void* rhs, void* out, int64_t m, int64_t k,
                        int64_t n, const int32_t* group_sizes, int32_t g_total,
                        int32_t group_offset, int32_t g_local, const int32_t* limit,
                        rd_epilogue epi, int32_t* status, rd_stream_t stream);

/*
 * rd_ragged_dot_trans_rhs -- the trans_rhs form (input gradient dx).
 *   out[i, :] = lhs[i, :] @ rhs[j, :, :]^T for every row i of local group j.
 * Defined by SkyRL PR #867 (review comment on the trans_ragged_dot
 * backward: dx = ragged_dot(y, do, group_sizes, trans_rhs=True)).
 *
 *   lhs  [m, n] bf16 (the output gradient), rhs [g_local, k, n] bf16,
 *   out  [m, k] bf16.  Other arguments as rd_ragged_dot.
 * Requires k % 8 == 0, n % 8 == 0, 16-byte aligned pointers, no overlap.
 */
rd_status rd_ragged_dot_trans_rhs(const void* lhs, const void* rhs, void* out, int64_t m,
                                  int64_t k, int64_t n, const int32_t* group_sizes,
                                  int32_t g_total, int32_t group_offset, int32_t g_local,
                                  const int32_t* limit, int32_t* status, rd_stream_t stream);

/*
 * rd_ragged_dot_trans_rhs_glu_bwd -- dx of an expert FFN's down projection with
 * the SiLU-GLU backward fused into its epilogue.
 *   dh[i, c]         = sum_n d_out[i, n] * rhs[j, c, n]      (f32, never stored)
 *   g = fused[i, c], u = fused[i, f + c], e = exp(-g), den = 1 + e,
 *   sig = 1 / den, silu = g / den                           (f32)
 *   d_fused[i, c]     = bf16((dh * u) * (sig * (1 + g * (1 - sig))))   (d_gate)
 *   d_fused[i, f + c] = bf16(dh * silu)                                (d_up)
 *   with -0 stored as +0, for every row i of local group j; rows in [0, L)
 *   outside the local groups are +0 in both halves; rows >= L untouched.
 * Defined by SkyRL PR #867 (trans_rhs form of the backward) and MaxText PR
 * #5760 (commit message: the GLU backward writes [d_gate | d_up] in one pass,
 * recomputing the forward from the saved fused buffer).  Unlike running
 * rd_ragged_dot_trans_rhs then rd_glu_bwd, dh is used unrounded and never
 * goes to memory.  Accuracy: within one bf16 ulp of the exact value of the
 * formulas, plus the GEMM error of dh carried through them; the logistic is
 * evaluated as 1 / (1 + exp(-|g|)) on either side of 0, so gates far below
 * zero keep their tiny gradients.
 *
 *   d_out [m, n] bf16, rhs [g_local, f, n] bf16 (the down weights, forward
 *   h [m, f] @ rhs[j] [f, n]), fused [m, 2f] bf16, d_fused [m, 2f] bf16.
 *   Other arguments as rd_ragged_dot.
 * Requires f % 8 == 0, n % 8 == 0, 16-byte aligned pointers; d_fused must
 * not overlap any input.
 */
rd_status rd_ragged_dot_trans_rhs_glu_bwd(const void* d_out, const void* rhs, const void* fused,
                                          void* d_fused, int64_t m, int64_t f, int64_t n,
                                          const int32_t* group_sizes, int32_t g_total,
                                          int32_t group_offset, int32_t g_local,
                                          const int32_t* limit, int32_t* status,
                                          rd_stream_t stream);

/*
 * rd_trans_ragged_dot -- per-group weight gradient.
 *   out[j, :, :] = x[rows_j, :]^T @ y[rows_j, :] for each local group j;
 *   a group without rows (or whose rows all lie at or past L) gives zeros.
 * Defined by SkyRL PR #867 (_gpu_trans_ragged_dot_fwd: x [m, k], y [m, n],
 * f32 accumulation) and MaxText PR #5760 (commit message: the grouped
 * matmuls skip rows outside the groups and past limit).
 *
 *   x [m, k] bf16, y [m, n] bf16, out [g_local, k, n] bf16 (f32 accumulated).
 *   workspace        device scratch of at least the size rd_trans_ragged_dot_
 *                    workspace_size reports for the current device, 128-byte
 *                    aligned, or NULL.  With it the kernel builds, per group,
 *                    TMA descriptors whose rows are exactly the group's rows
 *                    (rows outside the group then arrive as zeros); without
 *                    it the rows of each group's first K block that precede
 *                    the group are zeroed in shared memory, which is slower
 *                    when group sizes are not multiples of 16.  The results
 *                    agree within the stated accuracy (only the f32
 *                    summation order differs).  The workspace is the call's
 *                    own until the call completes on its stream: calls that
 *                    may run at the same time need separate workspaces.  The
 *                    library never reads what the workspace held before.
 *   workspace_bytes  its size in bytes (ignored when workspace is NULL).
 *   Other arguments as rd_ragged_dot.
 * Requires k % 8 == 0, n % 8 == 0, 16-byte aligned pointers, no overlap
 * (the workspace included); RD_ERR_INVALID_ARG for a workspace that is too
 * small.
 */
rd_status rd_trans_ragged_dot(const void* x, const void* y, void* out, int64_t m, int64_t k,
                              int64_t n, const int32_t* group_sizes, int32_t g_total,
                              int32_t group_offset, int32_t g_local, const int32_t* limit,
                              void* workspace, size_t workspace_bytes, int32_t* status,
                              rd_stream_t stream);

/*
 * rd_trans_ragged_dot_workspace_size -- the workspace rd_trans_ragged_dot and
 * rd_trans_ragged_dot_f32 take on the current device: 2 KB per SM (the
 * per-group TMA descriptors of each CTA).  RD_ERR_INVALID_ARG for a NULL
 * pointer, RD_ERR_UNSUPPORTED on a device other than sm_103.
 */
rd_status rd_trans_ragged_dot_workspace_size(size_t* bytes);

/*
 * rd_trans_ragged_dot_f32 -- per-group weight gradient kept in f32, optionally
 * accumulated into the output (gradient accumulation across micro-batches).
 *   accumulate = 0: out[j] = x[rows_j]^T @ y[rows_j]   (a group without rows: zeros)
 *   accumulate = 1: out[j] += x[rows_j]^T @ y[rows_j]  (a group without rows: unchanged)
 * The sum is the tensor cores' f32 accumulation; the add of the accumulating
 * form rounds once, to nearest.  SkyRL PR #867 (_gpu_trans_ragged_dot_fwd
 * separates acc_dtype = f32 from the compute dtype).
 *
 *   x [m, k] bf16, y [m, n] bf16, out [g_local, k, n] f32.  Other arguments
 *   (the workspace included) as rd_trans_ragged_dot.  Calls that accumulate
 *   into the same buffer must be ordered on one stream.
 */
rd_status rd_trans_ragged_dot_f32(const void* x, const void* y, float* out, int64_t m, int64_t k,
                                  int64_t n, const int32_t* group_sizes, int32_t g_total,
                                  int32_t group_offset, int32_t g_local, const int32_t* limit,
                                  int32_t accumulate, void* workspace, size_t workspace_bytes,
                                  int32_t* status, rd_stream_t stream);

/*
 * rd_trans_ragged_dot_no_alloc -- rd_trans_ragged_dot for callers that cannot
 * allocate device memory.  The source pages have no counterpart: this entry
 * point exists for code that has no way to provide the workspace, such as a
 * caller running inside a memory allocator's own callbacks, a runtime that
 * owns every device allocation and hands out no scratch, or a process that
 * must not grow its footprint after set-up.  It computes what
 * rd_trans_ragged_dot computes with a workspace (the per-group-descriptor
 * form), taking its 2 KB of descriptors per SM from a 512 KB array inside the
 * library that every GPU loading the library holds until the process exits;
 * it allocates nothing and calls no allocating routine.
 *
 *   Arguments as rd_trans_ragged_dot, without the workspace.
 *   Limit: devices of up to 256 SMs; on a larger device it returns
 *   RD_ERR_UNSUPPORTED and enqueues nothing.
 *   Set-up: the first call on each device asks the CUDA runtime for the
 *   array's device address (once per device, with that device current); make
 *   that first call before any stream capture on the device.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's descriptors; no call reads what an earlier one left there.  Calls
 *   whose kernels overlap on the GPU (other streams, other threads) race on
 *   the array and give wrong results: order such calls on one stream.
 */
rd_status rd_trans_ragged_dot_no_alloc(const void* x, const void* y, void* out, int64_t m,
                                       int64_t k, int64_t n, const int32_t* group_sizes,
                                       int32_t g_total, int32_t group_offset, int32_t g_local,
                                       const int32_t* limit, int32_t* status, rd_stream_t stream);

/*
 * rd_glu_fwd -- SiLU-GLU forward over the valid rows of a fused buffer.
 *   out[r, c] = bf16( g / (1 + exp(-g)) * u ),  g = fused[r, c], u = fused[r, f + c],
 *   for r < L; rows >= L of out are not written and of fused not read.
 * Defined by MaxText PR #5760 (commit message, kernels/ragged/glu_rows.py:
 * gate and up read in place from the fused buffer, XLA's op sequence
 * negate, exp, +1, divide, multiply in f32, rounded only at the output).
 * Accuracy: within one bf16 ulp of the exact value; where that op sequence
 * gives an infinity, a NaN or (for g below -88.72, where exp(-g) overflows
 * binary32) a signed zero, the output has exactly its bits.
 *
 *   fused [rows, 2f] bf16, out [rows, f] bf16, limit device int32 or NULL.
 * Requires f % 8 == 0, 16-byte aligned pointers, out not overlapping fused.
 */
rd_status rd_glu_fwd(const void* fused, void* out, int64_t rows, int64_t f,
                     const int32_t* limit, rd_stream_t stream);

/*
 * rd_glu_bwd -- SiLU-GLU backward, writing [d_gate | d_up] in one pass.
 *   with g, u as above and d = d_out[r, c], in f32:
 *   e = exp(-g), den = 1 + e, sig = 1 / den, silu = g / den,
 *   d_fused[r, f + c] = bf16(d * silu),
 *   d_fused[r, c]     = bf16((d * u) * (sig * (1 + g * (1 - sig)))),
 *   and any result that rounds to -0 is stored as +0; rows r < L only.
 * Defined by MaxText PR #5760 (commit message: the backward writes
 * [d_gate | d_up] in one pass with the -0 -> +0 fix, recomputing the
 * forward from the saved fused buffer).  Accuracy as rd_glu_fwd: within one
 * bf16 ulp of the exact value, and the op sequence's bits wherever it gives
 * an infinity, a NaN or a zero from the overflow of exp(-g).
 *
 *   fused [rows, 2f] bf16, d_out [rows, f] bf16, d_fused [rows, 2f] bf16.
 * Requires f % 8 == 0, 16-byte aligned pointers, d_fused not overlapping
 * the inputs.
 */
rd_status rd_glu_bwd(const void* fused, const void* d_out, void* d_fused, int64_t rows,
                     int64_t f, const int32_t* limit, rd_stream_t stream);

/*
 * rd_unsort_bwd_rows -- valid-rows unsort backward.
 *   grad[r, :] = bf16( f32(g[r, :]) * w[r] )               (one f32 multiply, one rounding)
 *   dot[r]     = sum_c f32(g[r, c]) * f32(y[r, c])         (f32 accumulation)
 *   for r < L; rows >= L of grad and dot are not written, of g, y, w not read.
 * Defined by MaxText PR #5760 (commit message, kernels/ragged/unsort_bwd_rows.py:
 * the weighted gradient and the f32 routing-weight row dot over rows < limit;
 * review comment: the per-row dot must not be assembled by concurrent blocks).
 * Each row is owned by one warp, so the result has no cross-CTA race.
 *
 *   g [rows, hidden] bf16 (gathered gradient), y [rows, hidden] bf16 (sorted
 *   tokens), w [rows] f32 (routing weights), grad [rows, hidden] bf16,
 *   dot [rows] f32, limit device int32 or NULL.
 * Requires hidden % 8 == 0, 16-byte aligned bf16 pointers, 4-byte aligned
 * w and dot; grad and dot must not overlap the inputs.
 */
rd_status rd_unsort_bwd_rows(const void* g, const void* y, const float* w, void* grad, float* dot,
                             int64_t rows, int64_t hidden, const int32_t* limit,
                             rd_stream_t stream);

/*
 * rd_tuning -- process-wide overrides of the grouped-GEMM launch choices, for
 * measurements and tests.  No page defines them: they select among kernels
 * that compute the same result (within the documented accuracy), or bound
 * the kernels' waits.
 *
 *   gemm_variant     RD_VARIANT_AUTO: the library picks the CTA-pair kernel
 *                    (256-row tiles, cta_group::2) when the buffer holds at
 *                    least 512 rows per group on average, else the
 *                    single-CTA kernel (128-row tiles);  RD_VARIANT_SINGLE /
 *                    RD_VARIANT_PAIR force one of them (all three grouped
 *                    GEMMs).
 *   band_rows        rows per band of the forward / dx tile order (within a
 *                    band the CTAs sweep every output column block before the
 *                    next band starts, so the band's lhs rows stay in L2);
 *                    0 = the default, 6144.  Rounded down to whole tiles
 *                    (at least one).
 *   wait_timeout_ns  bound of every wait inside the grouped-GEMM kernels;
 *                    0 = the default, 4 s.
 *   reserved         must be 0 (room for later fields).
 *
 * The values apply to calls made after rd_set_tuning returns, from any
 * thread; a call reads them on the host when it builds its launch, so a
 * CUDA graph keeps the values that were in force when it was captured.
 * rd_set_tuning(NULL) restores the defaults.  Returns RD_ERR_INVALID_ARG
 * (and changes nothing) for an unknown variant, a negative band_rows or a
 * nonzero reserved field.
 */
#define RD_VARIANT_AUTO 0
#define RD_VARIANT_SINGLE 1
#define RD_VARIANT_PAIR 2

typedef struct {
  int32_t gemm_variant;
  int32_t band_rows;
  uint64_t wait_timeout_ns;
  int32_t reserved[2];
} rd_tuning;

rd_status rd_set_tuning(const rd_tuning* t);
/* The values in force (0 fields read back as 0, i.e. the defaults). */
rd_status rd_get_tuning(rd_tuning* t);

/* A static, human-readable name for a status code. */
const char* rd_status_string(rd_status s);

#ifdef __cplusplus
}
#endif

#endif /* RD_H_ */
