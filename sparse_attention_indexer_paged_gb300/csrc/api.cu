// C ABI of the indexer library: argument checks, tensor maps, launches.
// Every entry point is stream-ordered; nothing here allocates, frees or
// synchronises.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace dsa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device check, cached per device: sm_103 is the only compiled target.
std::atomic<int> g_dev_ok[64];

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DSA_ERR_NO_DEVICE;
  if (dev < 64) {
    const int cached = g_dev_ok[dev].load(std::memory_order_relaxed);
    if (cached == 1) return DSA_OK;
    if (cached == 2) return DSA_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return DSA_ERR_NO_DEVICE;
  const bool ok = major == 10 && minor == 3;
  if (dev < 64) g_dev_ok[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? DSA_OK : DSA_ERR_NO_DEVICE;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

}  // namespace

bool encode_tensor_map_u8(void* tmap_out, int rank, void* base, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
  if (swizzle_bytes != 0 && swizzle_bytes != 64 && swizzle_bytes != 128) return false;
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  const CUresult r = g_encode(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_UINT8,
                              static_cast<cuuint32_t>(rank), base, gd, gs, bx, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                              : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case DSA_ERR_SCHEDULE_MISMATCH: return "schedule was built for other rows, mode or SM count";
    case DSA_ERR_CUDA: return "CUDA runtime or launch error";
    case DSA_ERR_BAD_BLOCK: return "page id outside the pool or past the block table";
    case DSA_ERR_TIMEOUT: return "a pipeline wait ran out; the kernel returned early";
    case DSA_ERR_NO_DEVICE: return "no sm_103 device";
    case DSA_ERR_SCRATCH_TOO_SMALL: return "the step needs more than the library's fixed scratch array holds";
    default: return "unknown status";
  }
}

int dsa_version(void) { return 100; }

int64_t dsa_schedule_words(int32_t num_sms, int32_t num_rows) {
  if (num_sms < 1 || num_rows < 0) return -1;
  return SchedLayout(num_sms, num_rows).words;
}

int32_t dsa_device_num_sms(void) {
  const int st = check_device();
  if (st != DSA_OK) return -st;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -DSA_ERR_CUDA;
  return n;
}

int dsa_paged_mqa_logits_metadata(const int32_t* context_lens, const int32_t* indices,
                                  int32_t num_rows, int32_t block_kv, int32_t num_sms,
                                  int32_t* schedule, dsa_stream_t stream) {
  return dsa_paged_mqa_logits_metadata_for_keys(context_lens, indices, num_rows, block_kv, num_sms, DSA_KV_FP8,
                                                schedule, stream);
}

int dsa_paged_mqa_logits_metadata_for_keys(const int32_t* context_lens, const int32_t* indices,
                                           int32_t num_rows, int32_t block_kv, int32_t num_sms,
                                           int32_t kv_format, int32_t* schedule, dsa_stream_t stream) {
  if (num_rows < 0 || num_sms < 1 || schedule == nullptr) return DSA_ERR_INVALID_ARG;
  if (kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4 && kv_format != DSA_KV_MXFP4) return DSA_ERR_INVALID_ARG;
  if (num_rows > 0 && context_lens == nullptr) return DSA_ERR_INVALID_ARG;
  if (num_sms > 1023 || num_rows > kMaxScheduleRows) return DSA_ERR_UNSUPPORTED;
  if (block_kv != kPageTokens) return DSA_ERR_UNSUPPORTED;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_metadata(context_lens, indices, num_rows, num_sms, kv_format,
                                       schedule, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The logits call of decode (row-indexed block table) and of prefill (a
// block table per request, read through the rows' request ids).
int logits_call(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes,
                int64_t num_pages,
                int32_t kv_format, const float* weights, const int32_t* context_lens,
                const int32_t* block_table, int64_t block_table_stride, const int32_t* bt_rows,
                int32_t bt_num_rows, const int32_t* indices, const int32_t* schedule, int32_t num_sms,
                void* logits, int32_t logits_dtype, int64_t logits_stride, int32_t num_rows,
                int32_t num_heads, int32_t head_dim, int32_t block_kv, int32_t* status,
                dsa_stream_t stream) {
  if (num_heads != kHeads || head_dim != kHeadDim || block_kv != kPageTokens)
    return DSA_ERR_UNSUPPORTED;
  if (kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4 && kv_format != DSA_KV_MXFP4) return DSA_ERR_UNSUPPORTED;
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || num_sms < 1 || num_sms > 1023) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!q || !kv_cache || !weights || !context_lens || !block_table || !schedule || !logits)
    return DSA_ERR_INVALID_ARG;
  // MXFP4 q comes with its ue8m0 scales; the other formats take e4m3 q alone
  if ((kv_format == DSA_KV_MXFP4) != (q_scale != nullptr) || (q_scale && !aligned(q_scale, 16)))
    return DSA_ERR_INVALID_ARG;
  const int64_t page_bytes = kv_format == DSA_KV_FP8   ? DSA_FP8_PAGE_BYTES
                             : kv_format == DSA_KV_FP4 ? DSA_FP4_PAGE_BYTES
                                                       : DSA_MXFP4_PAGE_BYTES;
  if (page_stride_bytes < page_bytes || page_stride_bytes % 16 != 0) return DSA_ERR_INVALID_ARG;
  if (num_pages < 1 || num_pages > INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (block_table_stride < 1 || logits_stride < 1 || logits_stride % 8 != 0 || logits_stride >= INT32_MAX)
    return DSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_rows) * kHeads >= (static_cast<int64_t>(1) << 31))
    return DSA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(weights, 16) || !aligned(logits, 16))
    return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  LogitsArgs a;
  a.q = static_cast<const uint8_t*>(q);
  a.q_scale = static_cast<const uint8_t*>(q_scale);
  a.kv_cache = static_cast<const uint8_t*>(kv_cache);
  a.page_stride = page_stride_bytes;
  a.num_pages = num_pages;
  a.kv_format = kv_format;
  a.weights = weights;
  a.context_lens = context_lens;
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.bt_rows = bt_rows;
  a.bt_num_rows = bt_num_rows;
  a.indices = indices;
  a.schedule = schedule;
  a.num_sms = num_sms;
  a.logits = logits;
  a.logits_dtype = logits_dtype;
  a.logits_stride = logits_stride;
  a.num_rows = num_rows;
  a.status = status;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = kv_format == DSA_KV_FP8   ? launch_logits_fp8(a, st)
                        : kv_format == DSA_KV_FP4 ? launch_logits_fp4(a, st)
                                                  : launch_logits_mxfp4(a, st);
  if (e == cudaErrorInvalidValue) return DSA_ERR_INVALID_ARG;
  if (e == cudaErrorNotSupported) return DSA_ERR_UNSUPPORTED;
  return launch_status(e);
}

}  // namespace

extern "C" {

int dsa_fp8_fp4_paged_mqa_logits(const void* q, const void* kv_cache, int64_t page_stride_bytes,
                                 int64_t num_pages, int32_t kv_format, const float* weights,
                                 const int32_t* context_lens, const int32_t* block_table,
                                 int64_t block_table_stride, const int32_t* indices,
                                 const int32_t* schedule, int32_t num_sms, void* logits,
                                 int32_t logits_dtype, int64_t logits_stride, int32_t num_rows,
                                 int32_t num_heads, int32_t head_dim, int32_t block_kv,
                                 int32_t* status, dsa_stream_t stream) {
  return logits_call(q, nullptr, kv_cache, page_stride_bytes, num_pages, kv_format, weights, context_lens,
                     block_table, block_table_stride, nullptr, 0, indices, schedule, num_sms, logits, logits_dtype,
                     logits_stride, num_rows, num_heads, head_dim, block_kv, status, stream);
}

int dsa_mxfp4_paged_mqa_logits(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes,
                               int64_t num_pages, const float* weights, const int32_t* context_lens,
                               const int32_t* block_table, int64_t block_table_stride, const int32_t* indices,
                               const int32_t* schedule, int32_t num_sms, void* logits, int32_t logits_dtype,
                               int64_t logits_stride, int32_t num_rows, int32_t num_heads, int32_t head_dim,
                               int32_t block_kv, int32_t* status, dsa_stream_t stream) {
  if (num_rows > 0 && q_scale == nullptr) return DSA_ERR_INVALID_ARG;
  return logits_call(q, q_scale, kv_cache, page_stride_bytes, num_pages, DSA_KV_MXFP4, weights, context_lens,
                     block_table, block_table_stride, nullptr, 0, indices, schedule, num_sms, logits, logits_dtype,
                     logits_stride, num_rows, num_heads, head_dim, block_kv, status, stream);
}

int dsa_prefill_rows(const int32_t* cu_seqlen_ks, const int32_t* cu_seqlen_ke, int32_t num_rows,
                     const int32_t* local_cu_seq_lens, int32_t num_requests, int32_t* context_lens,
                     int32_t* request_ids, int32_t* status, dsa_stream_t stream) {
  if (num_rows < 0 || num_requests < 1) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!cu_seqlen_ks || !cu_seqlen_ke || !local_cu_seq_lens || !context_lens || !request_ids)
    return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_prefill_rows(cu_seqlen_ks, cu_seqlen_ke, num_rows, local_cu_seq_lens, num_requests,
                                           context_lens, request_ids, status,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int dsa_prefill_mqa_logits(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages,
                           int32_t kv_format, const float* weights, const int32_t* context_lens,
                           const int32_t* request_ids, const int32_t* block_table, int64_t block_table_stride,
                           int32_t num_requests, const int32_t* schedule, int32_t num_sms, void* logits,
                           int32_t logits_dtype, int64_t logits_stride, int32_t num_rows, int32_t num_heads,
                           int32_t head_dim, int32_t block_kv, int32_t* status, dsa_stream_t stream) {
  if (num_rows > 0 && (request_ids == nullptr || num_requests < 1)) return DSA_ERR_INVALID_ARG;
  return logits_call(q, q_scale, kv_cache, page_stride_bytes, num_pages, kv_format, weights, context_lens,
                     block_table, block_table_stride, request_ids, num_requests, request_ids, schedule, num_sms, logits,
                     logits_dtype, logits_stride, num_rows, num_heads, head_dim, block_kv, status, stream);
}

int dsa_top_k_per_row(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                      const int32_t* row_starts, const int32_t* row_ends, int32_t num_rows,
                      int32_t k, int32_t* out_idx, int64_t out_stride, int32_t* status,
                      dsa_stream_t stream) {
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || out_stride < k) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!logits || !row_ends || !out_idx) return DSA_ERR_INVALID_ARG;
  if (logits_stride < 1 || logits_stride % 4 != 0 || logits_stride >= INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 16)) return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_top_k(logits, logits_dtype, logits_stride, row_starts, row_ends,
                                    num_rows, k, out_idx, out_stride, status,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int dsa_dcp_pack_topk(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                      const int32_t* local_idx, int64_t idx_stride, int32_t num_rows, int32_t k,
                      int32_t dcp_rank, int32_t dcp_world, int32_t interleave, float* packed,
                      dsa_stream_t stream) {
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > DSA_MAX_TOPK || dcp_world < 1 || dcp_world > DSA_DCP_MAX_WORLD) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || idx_stride < k || dcp_rank < 0 || dcp_rank >= dcp_world || interleave < 1)
    return DSA_ERR_INVALID_ARG;
  if (logits_stride < 1 || logits_stride * dcp_world >= (int64_t{1} << 24)) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!logits || !local_idx || !packed || !aligned(packed, 8)) return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_dcp_pack(logits, logits_dtype, logits_stride, local_idx, idx_stride, num_rows, k,
                                       dcp_rank, dcp_world, interleave, packed,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int dsa_dcp_merge_topk(const float* gathered, int32_t dcp_world, int32_t num_rows, int32_t k,
                       int32_t* out_idx, int64_t out_stride, dsa_stream_t stream) {
  if (k < 1 || k > DSA_MAX_TOPK || dcp_world < 1 || dcp_world > DSA_DCP_MAX_WORLD) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || out_stride < k) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!gathered || !out_idx || !aligned(gathered, 8)) return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_dcp_merge(gathered, dcp_world, num_rows, k, out_idx, out_stride,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int dsa_selftest_wait_timeout(int64_t timeout_ns, int32_t* status, dsa_stream_t stream) {
  if (timeout_ns < 1000 || timeout_ns > 1000000000 || status == nullptr) return DSA_ERR_INVALID_ARG;
  const int dev = check_device();
  if (dev != DSA_OK) return dev;
  return launch_status(launch_selftest_wait(static_cast<uint64_t>(timeout_ns), status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
