// Shared constants and host-side launch declarations of the indexer library.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "dsa_indexer.h"

namespace dsa {

// Supported shape.
constexpr int kHeads = DSA_NUM_HEADS;       // 64
constexpr int kHeadDim = DSA_HEAD_DIM;      // 128
constexpr int kPageTokens = DSA_BLOCK_KV;   // 64 tokens per page

// Schedule: a tile is two pages (128 keys, the M of one MMA); runs of equal
// request ids are cut into groups of at most kGroupMaxRows rows; a unit is
// one tile of one group.  The metadata call orders the groups by row count,
// lays their units end to end and gives SM i the units between its two
// boundaries at both ends of that sequence (metadata.cu states the rule).
//
// Layout (int32 words):
//   header[8] = {kScheduleMagic, rows T, varlen flag, SMs S, groups G,
//                units U, kTileTokens, kGroupMaxRows}
//   left[S + 1]   SM i owns sorted units [left[i], left[i + 1]) ...
//   right[S + 1]  ... and [right[i + 1], right[i])
//   grs[T + 1]    first row of group g (row order); entries past G hold T
//   pos[T + 1]    sorted position k: first row of its group | rows << 24;
//                 entries past G hold T
//   sus[T + 1]    first unit of sorted position k; entries past G hold U
//   spp_lo[T + 1], spp_hi[T + 1]  weight (unit_weight) before position k
constexpr int kTileTokens = 128;
constexpr int kGroupMaxRows = 8;
// Rows a group holds for each key format: what one pass of that format's
// logits kernel over a tile serves (FP8 all 8; MXFP4 6, its last TMEM
// columns holding scale factors; FP4 4, converting q into a pass-sized
// buffer), so that a unit costs one pass.  The logits call takes a schedule
// of any group size up to kGroupMaxRows.
__host__ __device__ constexpr int group_rows_for(int kv_format) {
  return kv_format == DSA_KV_FP4 ? 4 : (kv_format == DSA_KV_MXFP4 ? 6 : kGroupMaxRows);
}
// What one unit (tile) of a group of `rows` rows weighs in the schedule's
// second balanced quantity (the first is the units themselves).  FP8 and
// MXFP4: 4n + n^2, since a tile's cost grows faster than its rows (a tile of
// 6 rows fills 6 of the 8 TMEM slots, so tiles no longer overlap; measured
// microseconds per FP8 tile by rows 0.49, 0.56, 0.65, 0.82, 1.01, 1.17; the
// MXFP4 kernel has the same pipeline and measured 9 us faster with this
// weight than with n); FP4: n, its tiles' cost being the conversion.
__host__ __device__ constexpr int64_t unit_weight(int kv_format, int rows) {
  return kv_format != DSA_KV_FP4 ? 4 * rows + rows * rows : rows;
}
constexpr int32_t kScheduleMagic = 0x44534132;
constexpr int kScheduleHeaderWords = 8;
constexpr int kPosRowsShift = 24;
constexpr int32_t kPosRowMask = (1 << kPosRowsShift) - 1;
constexpr int32_t kMaxScheduleRows = kPosRowMask;  // rows must fit the position words

struct SchedLayout {
  int64_t left, right, grs, pos, sus, spp_lo, spp_hi, words;
  __host__ __device__ SchedLayout(int64_t S, int64_t T) {
    left = kScheduleHeaderWords;
    right = left + (S + 1);
    grs = right + (S + 1);
    pos = grs + (T + 1);
    sus = pos + (T + 1);
    spp_lo = sus + (T + 1);
    spp_hi = spp_lo + (T + 1);
    words = spp_hi + (T + 1);
  }
};

// Device status codes (same values as dsa_status_t).
constexpr int kErrScheduleMismatch = DSA_ERR_SCHEDULE_MISMATCH;
constexpr int kErrBadBlock = DSA_ERR_BAD_BLOCK;
constexpr int kErrTimeout = DSA_ERR_TIMEOUT;
constexpr int kErrInvalid = DSA_ERR_INVALID_ARG;

// A pipeline wait that sees no progress for this long gives up (the kernel
// then records DSA_ERR_TIMEOUT and returns).  Draining in-flight copies before
// exit is bounded separately.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainTimeoutNs = 200000000ull;   // 0.2 s
// Longest a waiting thread sleeps inside one try_wait before it re-checks
// the abort flag and the clock (it wakes earlier when the phase completes).

// Launch `kernel` so that it may start while the kernel before it on the
// stream is still running (programmatic dependent launch): its blocks set up
// (barriers, TMEM) and then wait at grid_dep_wait() until that kernel has
// finished and its writes are visible.  The earlier kernel lets it start with
// grid_dep_launch(); without one it starts at that kernel's end.
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// ----------------------------------------------------------------- launchers
// (defined in the kernel translation units, called by api.cu after the
// arguments have been checked)

cudaError_t launch_metadata(const int32_t* context_lens, const int32_t* indices, int32_t num_rows,
                            int32_t num_sms, int32_t kv_format, int32_t* schedule, cudaStream_t stream);

struct LogitsArgs {
  const uint8_t* q;
  const uint8_t* q_scale = nullptr;  // MXFP4: ue8m0 [T][H][D/32]
  const uint8_t* kv_cache;
  int64_t page_stride;
  int64_t num_pages;
  int32_t kv_format;
  const float* weights;
  const int32_t* context_lens;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* bt_rows = nullptr;  // per-row block-table row (null: row-indexed table)
  int32_t bt_num_rows = 0;
  const int32_t* indices;
  const int32_t* schedule;
  int32_t num_sms;
  void* logits;
  int32_t logits_dtype;
  int64_t logits_stride;
  int32_t num_rows;
  int32_t* status;
};

cudaError_t launch_logits_fp8(const LogitsArgs& a, cudaStream_t stream);
cudaError_t launch_logits_fp4(const LogitsArgs& a, cudaStream_t stream);
cudaError_t launch_logits_mxfp4(const LogitsArgs& a, cudaStream_t stream);

cudaError_t launch_top_k(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                         const int32_t* row_starts, const int32_t* row_ends, int32_t num_rows,
                         int32_t k, int32_t* out_idx, int64_t out_stride, int32_t* status,
                         cudaStream_t stream);

cudaError_t launch_dcp_pack(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                            const int32_t* local_idx, int64_t idx_stride, int32_t num_rows, int32_t k,
                            int32_t rank, int32_t world, int32_t interleave, float* packed,
                            cudaStream_t stream);
cudaError_t launch_prefill_rows(const int32_t* ks, const int32_t* ke, int32_t num_rows, const int32_t* starts,
                                int32_t num_requests, int32_t* ctx, int32_t* req, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_dcp_merge(const float* gathered, int32_t world, int32_t num_rows, int32_t k,
                             int32_t* out_idx, int64_t out_stride, cudaStream_t stream);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, int32_t* status, cudaStream_t stream);

// Tensor-map encoding through the driver entry point (no libcuda link).
// swizzle_bytes: 0 (none), 64 or 128 (the inner box is that many bytes).
bool encode_tensor_map_u8(void* tmap_out, int rank, void* base, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);

}  // namespace dsa
