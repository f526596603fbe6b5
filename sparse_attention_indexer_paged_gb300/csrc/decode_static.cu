// The whole decode step (schedule, logits, top-k) for callers that cannot
// allocate device memory: its scratch lives in a fixed array of this
// library's device image instead of a caller-provided buffer.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not
// available - inside a custom allocator's own callbacks, in a plugin whose
// host framework owns every allocation and hands out only the tensors of the
// op, or on a serving path whose memory is fixed after start-up.  Those
// callers still pass inputs and outputs; only the step's intermediate logits
// and its schedule move here.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds it (kStaticScratchBytes) until the process exits.  Host code
// cannot use its name as a device address; the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int64_t kStaticScheduleWords = DSA_STATIC_SCHEDULE_WORDS;
constexpr int64_t kStaticScheduleBytes = kStaticScheduleWords * 4;
constexpr int64_t kStaticLogitsBytes = DSA_STATIC_LOGITS_BYTES;
constexpr int64_t kStaticScratchBytes = kStaticScheduleBytes + kStaticLogitsBytes;
static_assert(kStaticScheduleBytes % 256 == 0, "the logits part must stay 256-byte aligned");

// schedule words first, then the logits of one row slice
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up on the
// first call for that device).
int static_scratch(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DSA_ERR_NO_DEVICE;
  if (dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear it, so that the caller's next runtime call does not report it
      return DSA_ERR_CUDA;
    }
    g_static_ptr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_static_ptr[dev]);
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_indexer_decode_topk_static(const void* q, const void* q_scale, const void* kv_cache,
                                   int64_t page_stride_bytes, int64_t num_pages, int32_t kv_format,
                                   const float* weights, const int32_t* context_lens,
                                   const int32_t* block_table, int64_t block_table_stride,
                                   const int32_t* indices, int32_t num_rows, int32_t num_heads,
                                   int32_t head_dim, int32_t block_kv, int32_t num_sms,
                                   int32_t logits_dtype, int64_t logits_stride, int32_t k,
                                   int32_t* out_idx, int64_t out_stride, int32_t* status,
                                   dsa_stream_t stream) {
  uint8_t* scratch = nullptr;
  int st = static_scratch(&scratch);
  if (st != DSA_OK) return st;
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || num_sms < 1 || logits_stride < 1) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  // The slices are cut so that their logits fit the array's logits part; the
  // smallest slice is 16 rows (or all rows, when fewer), and its schedule must
  // fit the schedule part.
  const int64_t eb = logits_dtype == DSA_LOGITS_BF16 ? 2 : 4;
  const int64_t min_rows = num_rows < 16 ? num_rows : 16;
  if (min_rows * logits_stride * eb > kStaticLogitsBytes) return DSA_ERR_SCRATCH_TOO_SMALL;
  int64_t need_bytes = 0, need_words = 0;
  st = dsa_indexer_decode_scratch(num_rows, logits_dtype, logits_stride, kStaticLogitsBytes, num_sms,
                                  &need_bytes, &need_words);
  if (st != DSA_OK) return st;
  if (need_bytes > kStaticLogitsBytes || need_words > kStaticScheduleWords) return DSA_ERR_SCRATCH_TOO_SMALL;
  return dsa_indexer_decode_topk(q, q_scale, kv_cache, page_stride_bytes, num_pages, kv_format, weights,
                                 context_lens, block_table, block_table_stride, indices, num_rows, num_heads,
                                 head_dim, block_kv, num_sms, logits_dtype, logits_stride, kStaticLogitsBytes,
                                 scratch + kStaticScheduleBytes, kStaticLogitsBytes,
                                 reinterpret_cast<int32_t*>(scratch), kStaticScheduleWords, k, out_idx,
                                 out_stride, status, stream);
}

}  // extern "C"
