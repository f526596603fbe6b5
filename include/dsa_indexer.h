/*
 * dsa_indexer.h - C ABI of the GB300 (sm_103a) DeepSeek-sparse-attention
 * indexer decode path: varlen paged MQA logits followed by per-row top-k.
 *
 * Three calls make one indexer decode step, in stream order:
 *
 *   dsa_paged_mqa_logits_metadata  -> per-SM work schedule
 *   dsa_fp8_fp4_paged_mqa_logits   -> logits[t, s] for every row t
 *   dsa_top_k_per_row              -> the k best columns of every row
 *
 * Conventions shared by every call:
 *   - Pointers marked (device) are CUDA device pointers of the current device;
 *     the caller allocates, owns and frees every buffer.  The library never
 *     allocates, frees or synchronises; it only enqueues kernels on `stream`
 *     (0 = the legacy default stream).  Calls are asynchronous.
 *   - The return value reports host-side checks and launch errors
 *     (dsa_status_t).  Faults found on the device (a page id out of range, a
 *     schedule built for other inputs, a pipeline wait that ran out) are
 *     written to `*status` (device int32, may be NULL) with atomicCAS from 0,
 *     so the first one sticks; the caller zeroes it and reads it when it
 *     wants.  A device fault leaves the outputs unspecified but never hangs
 *     or traps the GPU.
 *   - Sizes: H = 64 heads, D = 128 head dim and block_kv = 64 tokens per page
 *     are the supported shape (others return DSA_ERR_UNSUPPORTED).
 *
 * Sources.  The operations are the ones named by the vLLM sparse attention
 * indexer pages:
 *   [PR47469] "[Attention][DSA] Route SM100 sparse-indexer decode through
 *             varlen paged MQA logits", Purpose and Changes;
 *   [PR56811] "[Bugfix][GLM-5.3-Flash] Fix fp8_fp4_paged_mqa_logits MQA kpool
 *             varlen path for speculative decode", Purpose;
 *   [DOCS]    vllm.model_executor.layers.sparse_attn_indexer API docs,
 *             sections _varlen_decode_rows, as_fp32_logits, forward_cpu,
 *             forward_cuda, kv_cache_as_quant_view, _gather_workspace_shapes.
 */
#ifndef DSA_INDEXER_H_
#define DSA_INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* = cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,       /* null pointer, negative size, misaligned buffer */
  DSA_ERR_UNSUPPORTED = 2,       /* H != 64, D != 128, block_kv != 64, k > 2048, ... */
  DSA_ERR_SCHEDULE_MISMATCH = 3, /* (device) schedule built for other rows / mode / SM count */
  DSA_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
  DSA_ERR_BAD_BLOCK = 5,         /* (device) page id outside [0, num_pages) or past the table */
  DSA_ERR_TIMEOUT = 6,           /* (device) a pipeline wait ran out; the kernel returned early */
  DSA_ERR_NO_DEVICE = 7,         /* no usable sm_103 device */
  DSA_ERR_SCRATCH_TOO_SMALL = 8  /* the step needs more than the library's fixed scratch array holds */
} dsa_status_t;

enum { DSA_KV_FP8 = 0, DSA_KV_FP4 = 1, DSA_KV_MXFP4 = 2 };
enum { DSA_LOGITS_F32 = 0, DSA_LOGITS_BF16 = 1 };

/* Tokens per page, heads and head dimension of the supported shape. */
#define DSA_BLOCK_KV 64
#define DSA_NUM_HEADS 64
#define DSA_HEAD_DIM 128
/* Bytes of one page: FP8 = 64 x 128 e4m3 codes, then 64 fp32 scales;
   FP4 = 64 x 64 bytes of packed e2m1 (element 2i in the low nibble of byte i),
   then 64 x 8 e4m3 block scales (one per 16 elements), then 64 fp32 token
   scales.  The page stride may be larger (a per-layer view into a shared
   allocation, [DOCS] forward_cpu) and must be a multiple of 16. */
#define DSA_FP8_PAGE_BYTES 8448
#define DSA_FP4_PAGE_BYTES 4864
/* MXFP4 page: packed e2m1 [64][64 B] then ue8m0 block scales [64][4] (block 32) */
#define DSA_MXFP4_PAGE_BYTES 4352
/* Largest k of dsa_top_k_per_row. */
#define DSA_MAX_TOPK 2048
/* Largest decode-context-parallel world the merge accepts. */
#define DSA_DCP_MAX_WORLD 8

/* Text of a status code (static storage). */
const char* dsa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dsa_version(void);

/* Number of int32 words of a schedule for `num_sms` SMs and `num_rows` rows:
   8 + 2 * (num_sms + 1) + 5 * (num_rows + 1). */
int64_t dsa_schedule_words(int32_t num_sms, int32_t num_rows);

/* SM count of the current device (what the metadata call should balance
   over), or a negative dsa_status_t. */
int32_t dsa_device_num_sms(void);

/*
 * dsa_paged_mqa_logits_metadata - per-SM work schedule of the logits call.
 *
 * [PR47469] Purpose/Changes: get_paged_mqa_logits_metadata(seq_lens,
 * block_kv, num_sms, indices) builds the SM schedule; passing the per-row
 * request id `indices` selects the varlen schedule.  [DOCS]
 * _varlen_decode_rows: a slice of rows gets its own schedule, built from that
 * slice's seq_lens and indices.
 *
 *   context_lens (device) int32 [num_rows]: causal limit L_t of each row
 *                (the row sees keys 0 .. L_t - 1); non-decreasing within a
 *                request.
 *   indices      (device) int32 [num_rows] or NULL: request id of each row.
 *                Rows of one request must be adjacent ([PR56811] Purpose).
 *                NULL means every row is its own request (plain decode;
 *                equal to indices = arange(num_rows)).
 *   num_rows     0 .. 2^24 - 1 (else DSA_ERR_UNSUPPORTED).
 *   block_kv     must be 64.
 *   num_sms      1 .. 1023 (normally dsa_device_num_sms()); the logits call
 *                must be given the same value.
 *   schedule     (device) int32 [dsa_schedule_words(num_sms, num_rows)], out.
 *
 * Rule (the pages fix the purpose, not the split; this is the library's):
 * runs of equal ids are cut into groups of at most 8 rows (this call; see
 * dsa_paged_mqa_logits_metadata_for_keys for other sizes); a unit is one
 * 128-key tile of a group (ceil(max L_t / 128) units per group) and costs its
 * SM one K tile from HBM plus MMA and epilogue work that grows with the
 * group's rows n: the unit weighs 4n + n^2 here and for MXFP4 keys (a tile's
 * cost grows faster than its rows), and n for the FP4 schedule of
 * dsa_paged_mqa_logits_metadata_for_keys.  The groups are ordered by row
 * count (stable) and their units laid end to end; SM i takes units from both
 * ends of that sequence, so that every SM owns floor or ceil of
 * units / num_sms units and, as nearly as the group sizes allow, the same
 * weight.  Layout:
 * header[8] = {0x44534132, num_rows, varlen flag, num_sms, num_groups,
 * num_units, 128, group rows (8 here)}, left[num_sms + 1], right[num_sms + 1] (SM i owns sorted
 * units [left[i], left[i+1]) and [right[i+1], right[i])),
 * group_row_start[num_rows + 1], position[num_rows + 1] (first row of the
 * group at sorted position k | its rows << 24), unit_start[num_rows + 1],
 * weight_before low and high words [num_rows + 1] each (the weight of the
 * units before position k); entries past the last group hold num_rows,
 * num_rows, num_units and the weight total.
 */
int dsa_paged_mqa_logits_metadata(const int32_t* context_lens, const int32_t* indices,
                                  int32_t num_rows, int32_t block_kv, int32_t num_sms,
                                  int32_t* schedule, dsa_stream_t stream);

/*
 * dsa_paged_mqa_logits_metadata_for_keys - the same schedule, with groups cut
 * at the rows one pass of the logits call serves for that key format:
 * DSA_KV_FP8 8 (= dsa_paged_mqa_logits_metadata), DSA_KV_MXFP4 6, DSA_KV_FP4 4
 * (an MXFP4 tile's pairs have 7 TMEM slots, and FP4 converts q into a
 * pass-sized buffer, so a larger group costs one pass per 6 or 4 rows while
 * the split counts it as one unit).
 * No counterpart in the pages, whose metadata call takes no key format; the
 * extra argument only sizes the groups (header word 7 records it).  Any
 * format's logits call accepts a schedule of any group size from 1 to 8;
 * this one balances the FP4 and MXFP4 calls better.
 *
 *   kv_format    DSA_KV_FP8, DSA_KV_FP4 or DSA_KV_MXFP4 (else
 *                DSA_ERR_INVALID_ARG); the other arguments and the layout are
 *                those of dsa_paged_mqa_logits_metadata.
 */
int dsa_paged_mqa_logits_metadata_for_keys(const int32_t* context_lens, const int32_t* indices,
                                           int32_t num_rows, int32_t block_kv, int32_t num_sms,
                                           int32_t kv_format, int32_t* schedule, dsa_stream_t stream);

/*
 * dsa_fp8_fp4_paged_mqa_logits - varlen paged MQA logits.
 *
 * [PR47469] Purpose and [PR56811] Purpose: rows that share a request id are
 * processed together, so one K page serves all of a request's rows and heads
 * with no padding to (B, max_decode_len).  [DOCS] _varlen_decode_rows: the
 * call takes q, weights, the key cache, seq_lens, the row-sliced block table,
 * the schedule and indices; [DOCS] forward_cuda: the FP8 q's per-token scale
 * is folded into the weights.
 *
 *   logits[t, s] = kscale[s] * sum_h weights[t, h] * max(0, sum_d q[t,h,d] * k[s,d])
 *                  for s < L_t;  -inf for L_t <= s < round_up(L_t, 64).
 *   FP8 keys: k[s, d] = e4m3 code; kscale[s] = the page's fp32 scale.
 *   FP4 keys: k[s, d] = e2m1 * e4m3 block scale of d / 16; kscale[s] = the
 *             page's fp32 token scale.
 *   Columns from round_up(L_t, 64) up to round_up(L_max, 64) (clipped to the
 *   stride), L_max the largest causal limit of the row's group (up to 8
 *   adjacent rows of one request), may also be written as -inf; columns past
 *   that are not written.
 *
 *   q            (device) e4m3 [num_rows][64][128], 16-byte aligned.
 *   kv_cache     (device) page pool, 16-byte aligned; page p at
 *                kv_cache + p * page_stride_bytes.
 *   page_stride_bytes >= page bytes of kv_format, multiple of 16.
 *   num_pages    pages in the pool, >= 1.
 *   kv_format    DSA_KV_FP8 or DSA_KV_FP4 (DSA_KV_MXFP4 keys take MXFP4 q:
 *                dsa_mxfp4_paged_mqa_logits; here they are DSA_ERR_INVALID_ARG).
 *   weights      (device) fp32 [num_rows][64], 16-byte aligned.
 *   context_lens (device) int32 [num_rows] (as for the metadata call).
 *   block_table  (device) int32 [num_rows][block_table_stride]: page ids of
 *                each row's keys.  Rows of one request must hold the same
 *                page ids; the kernel reads them from the last row of each
 *                group (the row with the largest causal limit).  Entries
 *                read must lie in [0, num_pages) and below the stride;
 *                others are reported as DSA_ERR_BAD_BLOCK.
 *   indices      (device) int32 [num_rows] or NULL; must be NULL exactly when
 *                the schedule was built with NULL (else
 *                DSA_ERR_SCHEDULE_MISMATCH, the kpool fault of [PR56811]).
 *   schedule     (device) output of the metadata call for these rows.
 *   num_sms      the num_sms the schedule was built for; one CTA per SM.
 *   logits       (device) fp32 or bf16 [num_rows][logits_stride], 16-byte
 *                aligned; logits_stride >= round_up(max L_t, 64) elements and
 *                a multiple of 8.
 *   logits_dtype DSA_LOGITS_F32 or DSA_LOGITS_BF16 (round to nearest even).
 *   num_heads, head_dim, block_kv: must be 64, 128, 64.
 */
int dsa_fp8_fp4_paged_mqa_logits(const void* q, const void* kv_cache, int64_t page_stride_bytes,
                                 int64_t num_pages, int32_t kv_format, const float* weights,
                                 const int32_t* context_lens, const int32_t* block_table,
                                 int64_t block_table_stride, const int32_t* indices,
                                 const int32_t* schedule, int32_t num_sms, void* logits,
                                 int32_t logits_dtype, int64_t logits_stride, int32_t num_rows,
                                 int32_t num_heads, int32_t head_dim, int32_t block_kv,
                                 int32_t* status, dsa_stream_t stream);

/*
 * dsa_mxfp4_paged_mqa_logits - the logits of the pages' own FP4 form: MXFP4
 * keys and q ([DOCS] kv_cache_as_quant_view and _gather_workspace_shapes: an
 * MXFP4 token is head_dim / 2 bytes of packed e2m1 and head_dim /
 * MXFP4_BLOCK_SIZE ue8m0 scales; forward_cuda: the FP4 q is a (values,
 * scales) pair).  Block size 32 (the OCP MX block).
 *
 *   logits[t, s] = sum_h weights[t, h] * max(0, sum_d q[t,h,d] * k[s,d]),
 *   q[t,h,d] = e2m1 * 2^(q_scale[t,h,d/32] - 127),
 *   k[s,d]   = e2m1 * 2^(page scale of (s, d/32) - 127)     (no token scale).
 *
 *   q        (device) packed e2m1 [num_rows][64][64], element 2i in the low
 *            nibble of byte i; 16-byte aligned.
 *   q_scale  (device) ue8m0 [num_rows][64][4], 16-byte aligned.
 *   kv_cache pages of DSA_MXFP4_PAGE_BYTES: packed e2m1 [64][64], then
 *            ue8m0 [64][4].
 * The other arguments, the -inf tail and the status word are those of
 * dsa_fp8_fp4_paged_mqa_logits.  The tensor core takes the packed e2m1
 * values and both operands' ue8m0 scales directly (block-scaled MMA,
 * kind::mxf4): every 32-element block product is formed exactly and scaled
 * by its two powers of two, the sum accumulated in fp32; a scale code 255
 * (NaN) on a block makes the logits that block enters non-finite.
 */
int dsa_mxfp4_paged_mqa_logits(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes,
                               int64_t num_pages, const float* weights, const int32_t* context_lens,
                               const int32_t* block_table, int64_t block_table_stride, const int32_t* indices,
                               const int32_t* schedule, int32_t num_sms, void* logits, int32_t logits_dtype,
                               int64_t logits_stride, int32_t num_rows, int32_t num_heads, int32_t head_dim,
                               int32_t block_kv, int32_t* status, dsa_stream_t stream);

/*
 * dsa_top_k_per_row - the k largest logits of each row.
 *
 * [DOCS] _varlen_decode_rows: selector(logits, seq_lens, ..., out, k) with the
 * rows' causal limits as row ends; [DOCS] forward_cpu: the output is pre-filled
 * with -1, which pads rows shorter than k; [DOCS] as_fp32_logits: BF16 logits
 * are upcast to fp32 for the selection, only below the row end (here the
 * upcast is exact and done while reading).
 *
 *   logits       (device) fp32 or bf16 [num_rows][logits_stride].
 *   row_starts   (device) int32 [num_rows] or NULL (= 0).
 *   row_ends     (device) int32 [num_rows]; columns [row_start, row_end) compete;
 *                row_end <= logits_stride.
 *   k            1 .. DSA_MAX_TOPK.
 *   out_idx      (device) int32 [num_rows][out_stride], out_stride >= k:
 *                the chosen columns in ascending order, then -1 up to k.
 *   status       (device) int32 or NULL: the selection has no device-side
 *                fault to report and never writes it.
 * Order: larger logit first; equal logits go to the lower column; -0 == +0;
 * NaN ranks below every number.  Needs no workspace: each row's working set
 * lives in its CTA's shared memory.
 */
int dsa_top_k_per_row(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                      const int32_t* row_starts, const int32_t* row_ends, int32_t num_rows,
                      int32_t k, int32_t* out_idx, int64_t out_stride, int32_t* status,
                      dsa_stream_t stream);

/*
 * dsa_dcp_pack_topk - packs one rank's local top-k for the decode context
 * parallel merge ([DOCS] _merge_dcp_topk_global: every rank holds 1/world of
 * each request's keys, scores them and takes a local top-k; the candidates
 * travel as (score, global token id) fp32 pairs).
 *
 * Shard mapping (the page names the interleave size; this is the reading):
 * keys go to ranks in blocks of `interleave` consecutive tokens, round robin,
 * so local position l of rank r holds global token
 * ((l / interleave) * world + r) * interleave + l % interleave.
 *
 *   logits       (device) fp32 or bf16 [num_rows][logits_stride]: this rank's
 *                local logits; logits_stride * world < 2^24 so that global
 *                ids are exact in fp32.
 *   local_idx    (device) int32 [num_rows][idx_stride]: this rank's top-k
 *                local columns (from dsa_top_k_per_row), -1 padded.
 *   k            1 .. DSA_MAX_TOPK; idx_stride >= k.
 *   dcp_rank, dcp_world, interleave: 0 <= rank < world <= DSA_DCP_MAX_WORLD,
 *                interleave >= 1.
 *   packed       (device) fp32 [num_rows][k][2]: (score, global id), or
 *                (-inf, -1) for a padded or out-of-range local column.
 */
int dsa_dcp_pack_topk(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                      const int32_t* local_idx, int64_t idx_stride, int32_t num_rows, int32_t k,
                      int32_t dcp_rank, int32_t dcp_world, int32_t interleave, float* packed,
                      dsa_stream_t stream);

/*
 * dsa_dcp_merge_topk - the global top-k from every rank's packed candidates
 * ([DOCS] _merge_dcp_topk_global: all-gather rank-major, then a stable top-k
 * over the candidates; a token in the global top-k has at most k - 1 tokens
 * above it, hence is in its own rank's local top-k, so the merge is exact).
 *
 *   gathered     (device) fp32 [dcp_world][num_rows][k][2], rank-major (the
 *                layout an all-gather along dim 0 of the packs produces).
 *   dcp_world    1 .. DSA_DCP_MAX_WORLD.
 *   out_idx      (device) int32 [num_rows][out_stride], out_stride >= k: the
 *                global ids of the k best candidates (larger score first,
 *                equal scores to the lower id, NaN below every number) in
 *                ascending order, then -1 up to k.  Candidates with id -1 are
 *                never chosen.
 *
 * Candidate ids are integers in [0, 2^24), distinct within a row (as
 * dsa_dcp_pack_topk writes them); their order inside the gathered rows is
 * free.  A repeated id is written once.  Returns DSA_ERR_UNSUPPORTED for k or
 * dcp_world out of range and DSA_ERR_INVALID_ARG for a null or misaligned
 * pointer or out_stride < k; the caller owns every buffer and nothing is
 * allocated.
 */
int dsa_dcp_merge_topk(const float* gathered, int32_t dcp_world, int32_t num_rows, int32_t k,
                       int32_t* out_idx, int64_t out_stride, dsa_stream_t stream);

/*
 * dsa_selftest_wait_timeout - exercises the failure path of the library's
 * kernels on the GPU without a fault.  The pages have no counterpart: this is
 * part of the library's own failure detection.
 *
 * Every pipeline wait in the kernels is bounded: a wait that sees no progress
 * for its time limit (2 s in the production kernels) records
 * DSA_ERR_TIMEOUT in the caller's status word, tells the other roles of its
 * CTA to stop, drains what it issued and returns, so the context stays
 * usable.  This call launches one small kernel that waits, with that same
 * code and a time limit of timeout_ns, on an mbarrier nothing arrives on.
 *
 *   timeout_ns  1e3 .. 1e9 (else DSA_ERR_INVALID_ARG).
 *   status      (device) int32; receives DSA_ERR_TIMEOUT (first error wins,
 *               as for the other calls).
 * Returns DSA_OK once launched; the status is valid after the stream
 * synchronises.
 */
int dsa_selftest_wait_timeout(int64_t timeout_ns, int32_t* status, dsa_stream_t stream);

/*
 * dsa_prefill_rows - prefill token rows over the paged cache ([DOCS] the CPU
 * indexer's prefill branch of forward_cpu: a prefill chunk lays its
 * requests' keys end to end, local_cu_seq_lens [B + 1] being the requests'
 * starts, and tags row t with cu_seqlen_ks[t], its request's start, and
 * cu_seqlen_ke[t], the end of the keys it sees).  Writes, per row, its
 * request (the last r with local_cu_seq_lens[r] <= ks, clamped to
 * [0, B - 1]; a length-0 row past the last start reads no key) and its
 * causal length ke - ks.  These are the context_lens and request_ids of
 * dsa_paged_mqa_logits_metadata (as indices) and dsa_prefill_mqa_logits.
 *
 *   cu_seqlen_ks, cu_seqlen_ke  (device) int32 [num_rows].
 *   local_cu_seq_lens           (device) int32 [num_requests + 1], non-decreasing.
 *   context_lens, request_ids   (device) int32 [num_rows], written.
 *   status                      (device, may be null) a negative length sets
 *                               DSA_ERR_INVALID_ARG there (the row gets 0).
 */
int dsa_prefill_rows(const int32_t* cu_seqlen_ks, const int32_t* cu_seqlen_ke, int32_t num_rows,
                     const int32_t* local_cu_seq_lens, int32_t num_requests, int32_t* context_lens,
                     int32_t* request_ids, int32_t* status, dsa_stream_t stream);

/*
 * dsa_prefill_mqa_logits - the logits of prefill rows, read straight from
 * the paged cache (the pages' prefill mqa_logits over their ragged
 * cu_seqlen_ks/ke, without gathering the keys): as dsa_fp8_fp4_paged_mqa_logits
 * with context_lens = ke - ks and a block table per request, block_table
 * [num_requests][block_table_stride], that row r reads through
 * request_ids[r].  The schedule comes from dsa_paged_mqa_logits_metadata on
 * (context_lens, request_ids); rows of a request must be adjacent.  Column s
 * of row t is the request's token s (0 <= s < ke - ks), -inf up to
 * round_up(ke - ks, 64); a request id outside [0, num_requests) sets
 * DSA_ERR_BAD_BLOCK in `status`.  q_scale is NULL, or the MXFP4 q scales
 * when kv_format is DSA_KV_MXFP4 (q then packed e2m1, as in
 * dsa_mxfp4_paged_mqa_logits).
 */
int dsa_prefill_mqa_logits(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages,
                           int32_t kv_format, const float* weights, const int32_t* context_lens,
                           const int32_t* request_ids, const int32_t* block_table, int64_t block_table_stride,
                           int32_t num_requests, const int32_t* schedule, int32_t num_sms, void* logits,
                           int32_t logits_dtype, int64_t logits_stride, int32_t num_rows, int32_t num_heads,
                           int32_t head_dim, int32_t block_kv, int32_t* status, dsa_stream_t stream);

/*
 * dsa_decode_chunk_ranges - host only: the row slices of a decode step whose
 * logits fit a byte budget ([DOCS] _decode_chunk_ranges: the rows are
 * independent; a slice is a whole number of 16-row units except the tail,
 * the slices are as few as the budget allows and as even as the units allow,
 * the larger ones first).
 *
 *   rows, width  rows and logits columns per row; a row costs 2 * width
 *                bytes (BF16 logits; pass 2 * stride for fp32 logits).
 *   budget       bytes, >= 0; 0 means no budget.
 *   ranges       (host) int32 [max_ranges][2]: (start, end) per slice.
 *   num_ranges   (host) receives the slice count; 0 means one pass over all
 *                rows (no rows, no budget, or everything fits).
 * DSA_ERR_INVALID_ARG for a negative budget or rows, width < 1, a budget
 * below 16 rows, or more slices than max_ranges.  No device is touched.
 */
int dsa_decode_chunk_ranges(int64_t rows, int64_t width, int64_t budget, int32_t* ranges,
                            int32_t max_ranges, int32_t* num_ranges);

/*
 * dsa_indexer_decode_scratch - host only: the sizes the caller allocates for
 * dsa_indexer_decode_topk, i.e. the logits of the largest slice and its
 * schedule.  The logits of a slice cost logits_stride bytes x 4 (fp32) or
 * x 2 (bf16) per row; the budget is counted in those bytes.
 */
int dsa_indexer_decode_scratch(int32_t num_rows, int32_t logits_dtype, int64_t logits_stride,
                               int64_t logits_budget, int32_t num_sms, int64_t* scratch_bytes,
                               int64_t* schedule_words);

/*
 * dsa_indexer_decode_topk - the whole decode step: for each row slice of
 * dsa_decode_chunk_ranges (or all rows when the logits fit the budget), the
 * slice's own schedule (dsa_paged_mqa_logits_metadata on the slice's rows,
 * as [DOCS] does for a row range of the varlen decode), its logits into the
 * caller's scratch, and its top-k into out_idx rows [start, end).
 *
 * Arguments are those of the three calls, for all rows; the slices are
 * pointer offsets into them (q_scale: NULL, or the MXFP4 q scales when
 * kv_format is DSA_KV_MXFP4).  logits_scratch and schedule hold at least what
 * dsa_indexer_decode_scratch returns and are reused by every slice (the
 * calls are stream-ordered).  Results equal one pass over all rows bit for
 * bit: a row's logits do not depend on the other rows.  Returns the first
 * error of the calls it issues; device faults go to `status`.
 */
int dsa_indexer_decode_topk(const void* q, const void* q_scale, const void* kv_cache, int64_t page_stride_bytes,
                            int64_t num_pages, int32_t kv_format, const float* weights,
                            const int32_t* context_lens, const int32_t* block_table,
                            int64_t block_table_stride, const int32_t* indices, int32_t num_rows,
                            int32_t num_heads, int32_t head_dim, int32_t block_kv, int32_t num_sms,
                            int32_t logits_dtype, int64_t logits_stride, int64_t logits_budget,
                            void* logits_scratch, int64_t scratch_bytes, int32_t* schedule,
                            int64_t schedule_words, int32_t k, int32_t* out_idx, int64_t out_stride,
                            int32_t* status, dsa_stream_t stream);

/* Sizes of the fixed device scratch array of dsa_indexer_decode_topk_static:
   schedule words, then logits bytes (8 MiB + 64 KiB in all, held by every GPU
   that loads the library until the process exits). */
#define DSA_STATIC_SCHEDULE_WORDS 16384
#define DSA_STATIC_LOGITS_BYTES 8388608

/*
 * dsa_indexer_decode_topk_static - dsa_indexer_decode_topk for callers that
 * cannot allocate device memory.  The pages have no counterpart: it exists
 * for code that runs where cudaMalloc is not allowed or not available (inside
 * an allocator's own callbacks, in a plugin whose framework owns every
 * allocation and passes only the op's tensors, on a serving path whose memory
 * is fixed after start-up).  Such a caller still passes every input and the
 * output; the step's intermediate logits and its schedule live in a fixed
 * array of the library's device image (DSA_STATIC_LOGITS_BYTES of logits,
 * DSA_STATIC_SCHEDULE_WORDS of schedule), and the call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments are those of dsa_indexer_decode_topk without the budget, scratch
 * and schedule buffers.  The rows run in slices whose logits fit the array
 * (the rule of dsa_decode_chunk_ranges with budget DSA_STATIC_LOGITS_BYTES);
 * the top-k equals dsa_indexer_decode_topk's bit for bit.
 *   DSA_ERR_SCRATCH_TOO_SMALL  when 16 rows of logits (all rows, if fewer)
 *                              exceed DSA_STATIC_LOGITS_BYTES
 *                              (logits_stride x 4 bytes a row for fp32, x 2
 *                              for bf16), or a slice's schedule exceeds
 *                              DSA_STATIC_SCHEDULE_WORDS; nothing is launched.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its
 * contents behind: nothing in it needs to start at zero (every word a call
 * reads, that call wrote first), but calls whose work overlaps on the GPU (two
 * streams, or two host threads on one device) race on it and must be ordered
 * by the caller.
 */
int dsa_indexer_decode_topk_static(const void* q, const void* q_scale, const void* kv_cache,
                                   int64_t page_stride_bytes, int64_t num_pages, int32_t kv_format,
                                   const float* weights, const int32_t* context_lens,
                                   const int32_t* block_table, int64_t block_table_stride,
                                   const int32_t* indices, int32_t num_rows, int32_t num_heads,
                                   int32_t head_dim, int32_t block_kv, int32_t num_sms,
                                   int32_t logits_dtype, int64_t logits_stride, int32_t k,
                                   int32_t* out_idx, int64_t out_stride, int32_t* status,
                                   dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H_ */
