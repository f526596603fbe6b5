// The whole decode step of the indexer (schedule, logits, top-k) as one host
// call, with the rows cut into slices whose logits fit a scratch budget
// (sparse_attn_indexer docs, _decode_chunk_ranges: rows are independent, so
// they are sliced in 16-row units, as few slices as the budget allows, as
// even as the units allow, the larger slices first so that one scratch sized
// for the first serves every slice; each slice gets its own schedule, as the
// varlen decode of a row range does there).
//
// Host code only: it issues the three stream-ordered calls per slice on
// pointer offsets and allocates nothing.
#include <cstdint>

#include "common.cuh"

namespace dsa {
namespace {

int logit_bytes(int32_t logits_dtype) { return logits_dtype == DSA_LOGITS_BF16 ? 2 : 4; }

// Slices of `rows` under `budget` bytes of BF16-sized logits of `width`
// columns: count == 0 means one pass over all rows.
struct SlicePlan {
  int64_t count = 0;
  int64_t base = 0;   // units of every slice
  int64_t extra = 0;  // the first `extra` slices hold one unit more
  int64_t rows = 0;

  int64_t start(int64_t i) const { return 16 * (i * base + (i < extra ? i : extra)); }
  int64_t end(int64_t i) const {
    const int64_t e = start(i) + 16 * (base + (i < extra ? 1 : 0));
    return e < rows ? e : rows;
  }
  int64_t largest() const { return count == 0 ? rows : end(0); }
};

int plan_slices(int64_t rows, int64_t width, int64_t budget, SlicePlan* p) {
  if (rows < 0 || rows > INT32_MAX || width < 1 || budget < 0) return DSA_ERR_INVALID_ARG;
  p->rows = rows;
  p->count = 0;
  if (rows == 0 || budget == 0) return DSA_OK;
  const int64_t row_bytes = 2 * width;           // one row of BF16 logits
  const int64_t fit = budget / row_bytes;        // rows the budget holds
  if (rows <= fit) return DSA_OK;                // everything fits: one pass
  const int64_t cap = fit / 16;                  // 16-row units a slice may hold
  if (cap < 1) return DSA_ERR_INVALID_ARG;       // not even 16 rows fit
  const int64_t units = (rows + 15) / 16;
  p->count = (units + cap - 1) / cap;
  p->base = units / p->count;
  p->extra = units % p->count;
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_decode_chunk_ranges(int64_t rows, int64_t width, int64_t budget, int32_t* ranges,
                            int32_t max_ranges, int32_t* num_ranges) {
  if (num_ranges == nullptr) return DSA_ERR_INVALID_ARG;
  *num_ranges = 0;
  SlicePlan p;
  const int st = plan_slices(rows, width, budget, &p);
  if (st != DSA_OK) return st;
  if (p.count > max_ranges || (p.count > 0 && ranges == nullptr)) return DSA_ERR_INVALID_ARG;
  for (int64_t i = 0; i < p.count; ++i) {
    ranges[2 * i] = static_cast<int32_t>(p.start(i));
    ranges[2 * i + 1] = static_cast<int32_t>(p.end(i));
  }
  *num_ranges = static_cast<int32_t>(p.count);
  return DSA_OK;
}

int dsa_indexer_decode_scratch(int32_t num_rows, int32_t logits_dtype, int64_t logits_stride,
                               int64_t logits_budget, int32_t num_sms, int64_t* scratch_bytes,
                               int64_t* schedule_words) {
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (!scratch_bytes || !schedule_words || num_sms < 1 || logits_stride < 1) return DSA_ERR_INVALID_ARG;
  SlicePlan p;
  const int64_t eb = logit_bytes(logits_dtype);
  const int st = plan_slices(num_rows, logits_stride * eb / 2, logits_budget, &p);
  if (st != DSA_OK) return st;
  const int64_t r = p.largest();
  *scratch_bytes = r * logits_stride * eb;
  *schedule_words = dsa_schedule_words(num_sms, static_cast<int32_t>(r));
  return DSA_OK;
}

int dsa_indexer_decode_topk(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes,
                            int64_t num_pages, int32_t kv_format, const float* weights,
                            const int32_t* context_lens, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* indices, int32_t num_rows,
                            int32_t num_heads, int32_t head_dim, int32_t block_kv, int32_t num_sms,
                            int32_t logits_dtype, int64_t logits_stride, int64_t logits_budget,
                            void* logits_scratch, int64_t scratch_bytes, int32_t* schedule,
                            int64_t schedule_words, int32_t k, int32_t* out_idx, int64_t out_stride,
                            int32_t* status, dsa_stream_t stream) {
  if (logits_dtype != DSA_LOGITS_F32 && logits_dtype != DSA_LOGITS_BF16) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (num_heads != kHeads || head_dim != kHeadDim || block_kv != kPageTokens) return DSA_ERR_UNSUPPORTED;
  if (num_rows < 0 || num_sms < 1 || logits_stride < 1 || out_stride < k) return DSA_ERR_INVALID_ARG;
  if (num_rows == 0) return DSA_OK;
  if (!q || !weights || !context_lens || !block_table || !logits_scratch || !schedule || !out_idx)
    return DSA_ERR_INVALID_ARG;
  if ((kv_format == DSA_KV_MXFP4) != (q_scale != nullptr)) return DSA_ERR_INVALID_ARG;
  const int64_t eb = logit_bytes(logits_dtype);
  SlicePlan p;
  int st = plan_slices(num_rows, logits_stride * eb / 2, logits_budget, &p);
  if (st != DSA_OK) return st;
  const int64_t largest = p.largest();
  if (scratch_bytes < largest * logits_stride * eb) return DSA_ERR_INVALID_ARG;
  if (schedule_words < dsa_schedule_words(num_sms, static_cast<int32_t>(largest))) return DSA_ERR_INVALID_ARG;
  const uint8_t* qb = static_cast<const uint8_t*>(q);
  const int64_t n = p.count == 0 ? 1 : p.count;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t s = p.count == 0 ? 0 : p.start(i);
    const int64_t e = p.count == 0 ? num_rows : p.end(i);
    const int32_t rows = static_cast<int32_t>(e - s);
    const int32_t* ctx = context_lens + s;
    const int32_t* ind = indices ? indices + s : nullptr;
    st = dsa_paged_mqa_logits_metadata_for_keys(ctx, ind, rows, block_kv, num_sms, kv_format, schedule, stream);
    if (st != DSA_OK) return st;
    if (kv_format == DSA_KV_MXFP4) {  // q: packed e2m1 with ue8m0 scales
      st = dsa_mxfp4_paged_mqa_logits(qb + s * int64_t{kHeads} * (kHeadDim / 2),
                                      static_cast<const uint8_t*>(q_scale) + s * int64_t{kHeads} * (kHeadDim / 32),
                                      kv_cache, page_stride_bytes, num_pages, weights + s * kHeads, ctx,
                                      block_table + s * block_table_stride, block_table_stride, ind, schedule,
                                      num_sms, logits_scratch, logits_dtype, logits_stride, rows, num_heads,
                                      head_dim, block_kv, status, stream);
    } else {
      st = dsa_fp8_fp4_paged_mqa_logits(qb + s * int64_t{kHeads} * kHeadDim, kv_cache, page_stride_bytes, num_pages,
                                        kv_format, weights + s * kHeads, ctx,
                                        block_table + s * block_table_stride, block_table_stride, ind, schedule,
                                        num_sms, logits_scratch, logits_dtype, logits_stride, rows, num_heads,
                                        head_dim, block_kv, status, stream);
    }
    if (st != DSA_OK) return st;
    st = dsa_top_k_per_row(logits_scratch, logits_dtype, logits_stride, nullptr, ctx, rows, k,
                           out_idx + s * out_stride, out_stride, status, stream);
    if (st != DSA_OK) return st;
  }
  return DSA_OK;
}

}  // extern "C"
