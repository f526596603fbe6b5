/*
 * CPU oracle for the DSA indexer decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads this file: it
 * is built and called by tests/, by __graft_entry__.smoke() (one small check)
 * and by bench.py's cpu_baseline / reference leg.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Everything here is the plain definition written out, in fp64, one element
 * at a time, with no blocking, fusion or reordering:
 *
 *   logits[t, s] = kscale[s] * sum_h w[t, h] * max(0, sum_d q[t, h, d] * k[s, d])
 *                  for s < L_t, and -inf for s >= L_t
 *
 * ("varlen paged MQA logits": PR 47469 "Route SM100 sparse-indexer decode
 * through varlen paged MQA logits", Purpose; the per-row causal limit and the
 * row-sliced block table follow the sparse_attn_indexer docs,
 * _varlen_decode_rows; the head-weighted ReLU score is the indexer score named
 * there as fp8_fp4_paged_mqa_logits.)  The key k[s, :] is read through the
 * row's block table, page = block_table[t][s / 64], slot = s % 64, and decoded
 * from its stored bits.
 *
 *   top_k_per_row: the k largest scores of columns [row_start, row_end), ties
 *   to the lower column, returned in ascending column order, padded with -1
 *   (sparse_attn_indexer docs: forward_cpu fills the top-k buffer with -1;
 *   _merge_dcp_topk_global names a stable top-k and -1 padding).
 *
 * Each function below cites the passage it follows.  Parity pins: see
 * tests/test_oracle_pins.py.  "parity unpinned" is stated beside any function
 * that has no pin (none at present).
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kKvFp8 = 0;
constexpr int kKvFp4 = 1;
constexpr int kKvMxfp4 = 2;

// Planted-mistake switch used only by the oracle's own pin tests, to show that
// every pin can fail.  0 = the correct definition.
int g_plant = 0;

// --- number formats --------------------------------------------------------

// OCP 8-bit floating point, E4M3 ("FN": no infinities, S.1111.111 is NaN):
// exponent bias 7, three mantissa bits, subnormals at exponent field 0.
double decode_e4m3(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int expo = (code >> 3) & 0xF;
  const int mant = code & 0x7;
  double mag;
  if (expo == 0xF && mant == 0x7) {
    return std::numeric_limits<double>::quiet_NaN();
  } else if (expo == 0) {
    mag = std::ldexp(static_cast<double>(mant) / 8.0, 1 - 7);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(mant) / 8.0, expo - 7);
  }
  return sign ? -mag : mag;
}

// OCP Microscaling FP4 E2M1: exponent bias 1, one mantissa bit, subnormal at
// exponent field 0, no NaN or infinity.
double decode_e2m1(uint8_t nibble) {
  const int sign = (nibble >> 3) & 1;
  const int expo = (nibble >> 1) & 0x3;
  const int mant = nibble & 0x1;
  double mag;
  if (expo == 0) {
    mag = static_cast<double>(mant) * 0.5;
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(mant) / 2.0, expo - 1);
  }
  return sign ? -mag : mag;
}

// OCP Microscaling E8M0 scale: 2^(code - 127); code 255 is NaN.
double decode_ue8m0(uint8_t code) {
  if (code == 0xFF) return std::numeric_limits<double>::quiet_NaN();
  return std::ldexp(1.0, static_cast<int>(code) - (g_plant == 13 ? 128 : 127));
}

float load_f32(const uint8_t* p) {
  float f;
  std::memcpy(&f, p, 4);
  return f;
}

// Decode the stored key of one token into fp64 values k[0..D) (without the
// per-token scale) and return the per-token scale.  Page layouts:
//   FP8: values [64][D] e4m3 at 0, fp32 scale[64] after the values.
//   FP4: packed e2m1 [64][D/2] at 0 (element 2i in the low nibble of byte i),
//        e4m3 block scales [64][D/16] after them, fp32 token scale[64] last.
//   MXFP4: packed e2m1 [64][D/2] at 0 (as FP4), then ue8m0 scales [64][D/32];
//        no token scale (it is 1).
// (Per-token payload: sparse_attn_indexer docs, _gather_workspace_shapes and
// kv_cache_as_quant_view -- MXFP4 is head_dim/2 packed bytes plus
// head_dim/MXFP4_BLOCK_SIZE ue8m0 scales, with the OCP MX block of 32; the
// split of values and scales inside the page and the two-level FP4 scale are
// the storage reading this oracle and its library share by definition.)
double decode_token(const uint8_t* page, int kv_format, int slot, int D, int block_kv,
                    double* k) {
  if (kv_format == kKvFp8) {
    const uint8_t* v = page + static_cast<int64_t>(slot) * D;
    for (int d = 0; d < D; ++d) k[d] = decode_e4m3(v[d]);
    return load_f32(page + static_cast<int64_t>(block_kv) * D + 4 * slot);
  }
  if (kv_format == kKvMxfp4) {
    const uint8_t* v = page + static_cast<int64_t>(slot) * (D / 2);
    const uint8_t* es = page + static_cast<int64_t>(block_kv) * (D / 2) + static_cast<int64_t>(slot) * (D / 32);
    for (int d = 0; d < D; ++d) {
      const uint8_t byte = v[d / 2];
      const uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      k[d] = decode_e2m1(nib) * decode_ue8m0(es[d / 32]);
    }
    return 1.0;
  }
  const uint8_t* v = page + static_cast<int64_t>(slot) * (D / 2);
  const uint8_t* bs = page + static_cast<int64_t>(block_kv) * (D / 2) +
                      static_cast<int64_t>(slot) * (D / 16);
  for (int d = 0; d < D; ++d) {
    const uint8_t byte = v[d / 2];
    const uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    const int blk = (g_plant == 6) ? (d / 32) : (d / 16);
    k[d] = decode_e2m1(nib) * decode_e4m3(bs[blk]);
  }
  return load_f32(page + static_cast<int64_t>(block_kv) * (D / 2 + D / 16) + 4 * slot);
}

template <typename F>
void parallel_for(int n, int nthreads, F&& fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 1 || n <= 1) {
    for (int i = 0; i < n; ++i) fn(i);
    return;
  }
  nthreads = std::min(nthreads, n);
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w) {
    pool.emplace_back([&, w]() {
      for (int i = w; i < n; i += nthreads) fn(i);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Status codes of the oracle's entry points.
enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,          // bad sizes or null pointers
  ORACLE_ERR_GROUPING = 2,     // equal request ids not adjacent
  ORACLE_ERR_CONTEXT = 3,      // a row's causal limit decreases inside a request, or < 0
  ORACLE_ERR_BLOCK_TABLE = 4,  // rows of one request read different pages
  ORACLE_ERR_BLOCK_ID = 5,     // a page id outside [0, num_pages)
  ORACLE_ERR_STRIDE = 6,       // logits row stride below round_up(max L_t, block_kv)
};

int oracle_version(void) { return 1; }

void oracle_set_plant(int p) { g_plant = p; }

double oracle_e4m3_value(uint8_t code) { return decode_e4m3(code); }

double oracle_e2m1_value(uint8_t nibble) { return decode_e2m1(nibble & 0xF); }

double oracle_ue8m0_value(uint8_t code) { return decode_ue8m0(code); }

// Preconditions of the varlen decode call (PR 56811 "Fix
// fp8_fp4_paged_mqa_logits MQA kpool varlen path for speculative decode",
// Purpose: consecutive equal request indices identify the rows of one
// request; sparse_attn_indexer docs, _varlen_decode_rows: block table sliced
// by row).  Rows of one request must be adjacent, see non-decreasing causal
// limits, and read the same pages; every page a row reads must exist; the
// logits row stride must hold round_up(L_t, block_kv) columns.
int oracle_validate(const int32_t* context_lens, const int32_t* indices,
                    const int32_t* block_table, int64_t bt_stride, int32_t num_rows,
                    int64_t num_pages, int32_t block_kv, int64_t logits_stride) {
  if (num_rows < 0 || block_kv <= 0 || (num_rows > 0 && (!context_lens || !block_table)))
    return ORACLE_ERR_ARG;
  int64_t max_pages_needed = 0;
  for (int t = 0; t < num_rows; ++t) {
    if (context_lens[t] < 0) return ORACLE_ERR_CONTEXT;
    const int64_t pages = (static_cast<int64_t>(context_lens[t]) + block_kv - 1) / block_kv;
    max_pages_needed = std::max(max_pages_needed, pages);
    if (pages > bt_stride) return ORACLE_ERR_ARG;
    for (int64_t p = 0; p < pages; ++p) {
      const int32_t b = block_table[t * bt_stride + p];
      if (b < 0 || b >= num_pages) return ORACLE_ERR_BLOCK_ID;
    }
    if (static_cast<int64_t>(context_lens[t]) > logits_stride) return ORACLE_ERR_STRIDE;
    if ((static_cast<int64_t>(context_lens[t]) + block_kv - 1) / block_kv * block_kv >
        logits_stride)
      return ORACLE_ERR_STRIDE;
  }
  if (!indices) return ORACLE_OK;
  // adjacency: a request id, once its run ends, never appears again
  std::vector<int32_t> seen;
  for (int t = 0; t < num_rows; ++t) {
    const bool new_run = (t == 0) || indices[t] != indices[t - 1];
    if (new_run) {
      if (std::find(seen.begin(), seen.end(), indices[t]) != seen.end())
        return ORACLE_ERR_GROUPING;
      seen.push_back(indices[t]);
    } else {
      if (context_lens[t] < context_lens[t - 1]) return ORACLE_ERR_CONTEXT;
      // rows of one request read identical pages over the longer row's span
      const int64_t pages = (static_cast<int64_t>(context_lens[t]) + block_kv - 1) / block_kv;
      int t0 = t - 1;
      while (t0 > 0 && indices[t0 - 1] == indices[t]) --t0;
      for (int64_t p = 0; p < pages; ++p) {
        if (block_table[t * bt_stride + p] != block_table[t0 * bt_stride + p])
          return ORACLE_ERR_BLOCK_TABLE;
      }
    }
  }
  (void)max_pages_needed;
  return ORACLE_OK;
}

// Paged MQA logits in fp64 (definition in the header comment).
//   q        [num_rows][H][D] e4m3 codes; with q_scale (MXFP4 keys only, the
//            pages' FP4 path quantises q with scales too: sparse_attn_indexer
//            docs, forward_cuda), packed e2m1 [num_rows][H][D/2] and q_scale
//            ue8m0 [num_rows][H][D/32]
//   weights  [num_rows][H] fp32 (the per-token q scale is folded into them:
//            sparse_attn_indexer docs, SparseAttnIndexer.forward_cuda)
//   rows     which rows to evaluate (NULL: all rows, in order); output row i
//            holds row rows[i]
//   logits   [n_sel][out_cols] fp64; columns >= L_t are -inf
//   bound    [n_sel][out_cols] fp64 or NULL: kscale * sum_h sum_d |w q k|, the
//            magnitude the accuracy tolerance is stated against
int oracle_paged_mqa_logits(const uint8_t* q, const uint8_t* q_scale, const uint8_t* kv_cache, int64_t page_stride,
                            int64_t num_pages, int32_t kv_format, const float* weights,
                            const int32_t* context_lens, const int32_t* block_table,
                            int64_t bt_stride, int32_t num_rows, int32_t H, int32_t D,
                            int32_t block_kv, const int32_t* rows, int32_t n_sel,
                            double* logits, double* bound, int64_t out_cols,
                            int32_t nthreads) {
  if (!q || !kv_cache || !weights || !context_lens || !block_table || !logits) return ORACLE_ERR_ARG;
  if (H <= 0 || D <= 0 || D % 32 != 0 || block_kv <= 0 || num_rows < 0) return ORACLE_ERR_ARG;
  if (kv_format != kKvFp8 && kv_format != kKvFp4 && kv_format != kKvMxfp4) return ORACLE_ERR_ARG;
  if ((kv_format == kKvMxfp4) != (q_scale != nullptr)) return ORACLE_ERR_ARG;
  if (n_sel < 0) return ORACLE_ERR_ARG;
  const int n_eval = rows ? n_sel : num_rows;
  for (int i = 0; i < n_eval; ++i) {
    const int t = rows ? rows[i] : i;
    if (t < 0 || t >= num_rows) return ORACLE_ERR_ARG;
    if (context_lens[t] < 0 || context_lens[t] > out_cols) return ORACLE_ERR_STRIDE;
    const int64_t pages = (static_cast<int64_t>(context_lens[t]) + block_kv - 1) / block_kv;
    for (int64_t p = 0; p < pages; ++p) {
      const int32_t b = block_table[t * bt_stride + p];
      if (b < 0 || b >= num_pages) return ORACLE_ERR_BLOCK_ID;
    }
  }
  const double neg_inf = -std::numeric_limits<double>::infinity();
  // Work items are (selected row, block of kColBlock columns); each output
  // element is computed on its own, so the split changes no arithmetic.
  constexpr int64_t kColBlock = 2048;
  const int64_t blocks_per_row = (out_cols + kColBlock - 1) / kColBlock;
  const int64_t n_items = static_cast<int64_t>(n_eval) * std::max<int64_t>(blocks_per_row, 1);
  parallel_for(static_cast<int>(n_items), nthreads, [&](int item) {
    const int i = static_cast<int>(item / std::max<int64_t>(blocks_per_row, 1));
    const int64_t c0 = (item % std::max<int64_t>(blocks_per_row, 1)) * kColBlock;
    const int64_t c1 = std::min<int64_t>(c0 + kColBlock, out_cols);
    const int t = rows ? rows[i] : i;
    const int32_t L = context_lens[t];
    std::vector<double> qd(static_cast<size_t>(H) * D), k(D);
    for (int64_t j = 0; j < static_cast<int64_t>(H) * D; ++j) {
      if (q_scale == nullptr) {
        qd[j] = decode_e4m3(q[static_cast<int64_t>(t) * H * D + j]);
      } else {  // MXFP4 q: packed e2m1 [H][D/2] and ue8m0 scales [H][D/32] per row
        const uint8_t byte = q[(static_cast<int64_t>(t) * H * D + j) / 2];
        const uint8_t nib = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        qd[j] = decode_e2m1(nib) * decode_ue8m0(q_scale[(static_cast<int64_t>(t) * H * D + j) / 32]);
      }
    }
    double* out = logits + static_cast<int64_t>(i) * out_cols;
    double* bnd = bound ? bound + static_cast<int64_t>(i) * out_cols : nullptr;
    for (int64_t s = c0; s < c1; ++s) {
      if (s >= L) {
        out[s] = neg_inf;
        if (bnd) bnd[s] = 0.0;
        continue;
      }
      const int64_t col_page = (g_plant == 3) ? (s / (2 * block_kv)) : (s / block_kv);
      const int32_t page_id = block_table[t * bt_stride + col_page];
      const uint8_t* page = kv_cache + static_cast<int64_t>(page_id) * page_stride;
      const int slot = static_cast<int>(s % block_kv);
      const double kscale = decode_token(page, kv_format, slot, D, block_kv, k.data());
      double acc = 0.0, mag = 0.0;
      for (int h = 0; h < H; ++h) {
        const double w = weights[static_cast<int64_t>(t) * H + h];
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
          const double qv = (g_plant == 1) ? qd[static_cast<int64_t>(d % H) * D + h % D]
                                           : qd[static_cast<int64_t>(h) * D + d];
          dot += qv * k[d];
          mag += std::fabs(w * qv * k[d]);
        }
        if (g_plant == 2) {
          acc += w * dot;                       // ReLU dropped
        } else if (g_plant == 4) {
          acc += w * std::max(-dot, 0.0);       // sign flipped inside ReLU
        } else if (g_plant == 5) {
          acc += std::max(dot, 0.0);            // head weight dropped
        } else {
          acc += w * std::max(dot, 0.0);
        }
      }
      out[s] = kscale * acc;
      if (bnd) bnd[s] = std::fabs(kscale) * mag;
    }
  });
  return ORACLE_OK;
}

// Per-row top-k (sparse_attn_indexer docs: _varlen_decode_rows calls the
// selector with the row ends = the rows' causal limits; forward_cpu pre-fills
// -1; _merge_dcp_topk_global: stable top-k, -1 padding).  Order: score
// descending, then column ascending (ties to the lower column); -0 equals +0;
// NaN ranks below every number.  The chosen columns are written in ascending
// column order, then -1 up to k.
//   scores    [num_rows][stride] fp64 (fp32 / bf16 logits convert exactly)
//   row_starts NULL means 0
int oracle_top_k_per_row(const double* scores, int64_t stride, const int32_t* row_starts,
                         const int32_t* row_ends, int32_t num_rows, int32_t k,
                         int32_t* out_idx, int64_t out_stride, int32_t nthreads) {
  if (!scores || !row_ends || !out_idx || k <= 0 || out_stride < k || num_rows < 0)
    return ORACLE_ERR_ARG;
  for (int t = 0; t < num_rows; ++t) {
    const int64_t a = row_starts ? row_starts[t] : 0;
    const int64_t b = row_ends[t];
    if (a < 0 || b > stride || (b > a && a >= stride)) return ORACLE_ERR_ARG;
  }
  parallel_for(num_rows, nthreads, [&](int t) {
    const int64_t a = row_starts ? row_starts[t] : 0;
    const int64_t b = std::max<int64_t>(row_ends[t], a);
    const double* row = scores + static_cast<int64_t>(t) * stride;
    std::vector<int64_t> cols;
    cols.reserve(static_cast<size_t>(b - a));
    for (int64_t s = a; s < b; ++s) cols.push_back(s);
    auto better = [&](int64_t x, int64_t y) {
      const double vx = row[x], vy = row[y];
      const bool nx = std::isnan(vx), ny = std::isnan(vy);
      if (nx || ny) return !nx && ny;
      if (g_plant == 7) return vx < vy;
      return vx > vy;
    };
    std::stable_sort(cols.begin(), cols.end(), better);
    const int64_t take = std::min<int64_t>(k, static_cast<int64_t>(cols.size()));
    std::vector<int64_t> chosen(cols.begin(), cols.begin() + take);
    std::sort(chosen.begin(), chosen.end());
    int32_t* out = out_idx + static_cast<int64_t>(t) * out_stride;
    for (int64_t i = 0; i < k; ++i) out[i] = i < take ? static_cast<int32_t>(chosen[i]) : -1;
  });
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// DCP (decode context parallelism): each rank holds 1/world of every
// request's keys and computes logits and a top-k over its shard; the ranks'
// top-k candidates are merged into the global top-k (sparse_attn_indexer
// docs, _merge_dcp_topk_global: pack (score, global id) per candidate,
// all-gather rank-major [world, rows, k, 2], stable top-k over the
// candidates; a token in the global top-k is in its owner's local top-k, so
// the merge is exact).
//
// Readings (the page names the interleave size and the packed layout but
// does not print the mapping or the output order):
//   * keys go to ranks in blocks of `interleave` consecutive tokens, round
//     robin: global token g lives on rank (g / I) mod world at local
//     position (g / (I * world)) * I + g mod I;
//   * a padded local slot (-1) packs as (-inf, -1) and is never chosen;
//   * the merged row is the global top-k in this library's top-k order:
//     larger score first, equal scores to the lower global id, NaN below
//     every number; the chosen ids in ascending order, then -1 up to k.
// ---------------------------------------------------------------------------
int64_t oracle_dcp_global_id(int64_t local, int32_t rank, int32_t world, int32_t interleave) {
  if (local < 0 || world < 1 || interleave < 1 || rank < 0 || rank >= world) return -1;
  const int64_t I = interleave;
  return ((local / I) * world + rank) * I + local % I;
}

int64_t oracle_dcp_local_len(int64_t len, int32_t rank, int32_t world, int32_t interleave) {
  if (len <= 0 || world < 1 || interleave < 1 || rank < 0 || rank >= world) return 0;
  int64_t n = 0;  // count the global tokens below len that live on `rank`
  for (int64_t g = 0; g < len; ++g)
    if ((g / interleave) % world == rank) ++n;
  return n;
}

// packed[t][j] = (score of local column local_idx[t][j], its global id), or
// (-inf, -1) for a padded slot.
int oracle_dcp_pack(const double* local_scores, int64_t stride, const int32_t* local_idx,
                    int64_t idx_stride, int32_t num_rows, int32_t k, int32_t rank, int32_t world,
                    int32_t interleave, double* packed) {
  if (!local_scores || !local_idx || !packed || num_rows < 0 || k < 1 || idx_stride < k ||
      world < 1 || interleave < 1 || rank < 0 || rank >= world)
    return ORACLE_ERR_ARG;
  for (int t = 0; t < num_rows; ++t) {
    for (int j = 0; j < k; ++j) {
      const int32_t l = local_idx[static_cast<int64_t>(t) * idx_stride + j];
      double* o = packed + (static_cast<int64_t>(t) * k + j) * 2;
      if (l < 0 || l >= stride) {
        o[0] = -std::numeric_limits<double>::infinity();
        o[1] = -1.0;
      } else {
        o[0] = local_scores[static_cast<int64_t>(t) * stride + l];
        o[1] = static_cast<double>(oracle_dcp_global_id(l, rank, world, interleave));
      }
    }
  }
  return ORACLE_OK;
}

// gathered: [world][rows][k][2]; out: the global top-k ids of each row.
int oracle_dcp_merge(const double* gathered, int32_t world, int32_t num_rows, int32_t k,
                     int32_t* out_idx, int64_t out_stride) {
  if (!gathered || !out_idx || world < 1 || num_rows < 0 || k < 1 || out_stride < k)
    return ORACLE_ERR_ARG;
  for (int t = 0; t < num_rows; ++t) {
    std::vector<std::pair<double, int64_t>> cand;  // (score, global id)
    for (int r = 0; r < world; ++r)
      for (int j = 0; j < k; ++j) {
        const double* c = gathered + ((static_cast<int64_t>(r) * num_rows + t) * k + j) * 2;
        if (c[1] >= 0) cand.emplace_back(c[0], static_cast<int64_t>(c[1]));
      }
    auto better = [](const std::pair<double, int64_t>& x, const std::pair<double, int64_t>& y) {
      const bool nx = std::isnan(x.first), ny = std::isnan(y.first);
      if (nx != ny) return ny;  // a number before NaN
      if (!nx && x.first != y.first) return g_plant == 8 ? x.first < y.first : x.first > y.first;
      return g_plant == 9 ? x.second > y.second : x.second < y.second;
    };
    std::sort(cand.begin(), cand.end(), better);
    const int64_t take = std::min<int64_t>(k, static_cast<int64_t>(cand.size()));
    std::vector<int64_t> chosen;
    for (int64_t i = 0; i < take; ++i) chosen.push_back(cand[static_cast<size_t>(i)].second);
    std::sort(chosen.begin(), chosen.end());
    int32_t* out = out_idx + static_cast<int64_t>(t) * out_stride;
    for (int64_t i = 0; i < k; ++i) out[i] = i < take ? static_cast<int32_t>(chosen[static_cast<size_t>(i)]) : -1;
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Prefill rows over the paged cache (sparse_attn_indexer docs, the CPU
// indexer's prefill branch of forward_cpu): a prefill chunk tags each token
// row t with cu_seqlen_ks[t], the start of its request in the chunk's
// concatenated key range (local_cu_seq_lens[0..B]), and cu_seqlen_ke[t], the
// end of the keys it sees.  Its request is the last r with
// local_cu_seq_lens[r] <= ks (a sorted search to the right, minus one), its
// causal length is ke - ks, and it reads the keys through that request's
// block-table row; the logits are then the decode definition above with
// L_t = ke - ks.  A row whose request index falls outside [0, B) (possible
// only for a length-0 row at the very end) reads request B - 1: it touches no
// page.  Returns ORACLE_ERR_ARG for a negative length.
// ---------------------------------------------------------------------------
int oracle_prefill_rows(const int32_t* cu_seqlen_ks, const int32_t* cu_seqlen_ke, int32_t num_rows,
                        const int32_t* local_cu_seq_lens, int32_t num_requests, int32_t* context_lens,
                        int32_t* request_ids) {
  if (num_rows < 0 || num_requests < 1 || (num_rows > 0 && (!cu_seqlen_ks || !cu_seqlen_ke ||
                                                           !local_cu_seq_lens || !context_lens ||
                                                           !request_ids)))
    return ORACLE_ERR_ARG;
  for (int t = 0; t < num_rows; ++t) {
    const int32_t ks = cu_seqlen_ks[t], ke = cu_seqlen_ke[t];
    int32_t at_or_below = 0;  // offsets <= ks among the B + 1 request starts
    for (int r = 0; r <= num_requests; ++r)
      if (local_cu_seq_lens[r] <= ks) ++at_or_below;
    int32_t req = at_or_below - 1;
    if (req < 0) req = 0;
    if (req >= num_requests) req = num_requests - 1;
    if (ke - ks < 0) return ORACLE_ERR_ARG;
    request_ids[t] = req;
    context_lens[t] = g_plant == 12 ? ke : ke - ks;
  }
  return ORACLE_OK;
}

// ---------------------------------------------------------------------------
// Row chunking of the decode step under a logits budget (sparse_attn_indexer
// docs, _decode_chunk_ranges: the rows are independent, so they may be cut
// into slices whose BF16 logits, rows x width x 2 bytes, fit the budget; a
// slice is a whole number of 16-row units except for the tail, the slices
// are as few as the budget allows and as even as the units allow, the larger
// ones first).
//
// Returns the number of slices written to ranges[2 * i] (start),
// ranges[2 * i + 1] (end); 0 means one pass over all rows (no rows, a zero
// budget, or everything fits).  -ORACLE_ERR_ARG for a negative budget, a
// non-positive width, a budget below 16 rows, or more slices than max_ranges.
// ---------------------------------------------------------------------------
int64_t oracle_decode_chunk_ranges(int64_t rows, int64_t width, int64_t budget, int32_t* ranges,
                                   int64_t max_ranges) {
  if (budget < 0 || width < 1 || rows < 0) return -ORACLE_ERR_ARG;
  if (rows == 0 || budget == 0 || rows * width * 2 <= budget) return 0;
  const int64_t rows_per_slice = budget / (2 * width) / 16 * 16;  // the most rows a slice may hold
  if (rows_per_slice < 16) return -ORACLE_ERR_ARG;
  const int64_t units = g_plant == 10 ? rows / 16 : (rows + 15) / 16;  // 16-row units, the last partial
  const int64_t per = rows_per_slice / 16;                              // units a slice may hold
  const int64_t count = (units + per - 1) / per;                        // fewest slices
  if (count > max_ranges || !ranges) return -ORACLE_ERR_ARG;
  const int64_t base = units / count, extra = units % count;            // the first `extra` get one more
  int64_t start = 0;
  for (int64_t i = 0; i < count; ++i) {
    const bool more = g_plant == 11 ? i >= count - extra : i < extra;
    const int64_t end = std::min(rows, start + 16 * (base + (more ? 1 : 0)));
    ranges[2 * i] = static_cast<int32_t>(start);
    ranges[2 * i + 1] = static_cast<int32_t>(end);
    start = end;
  }
  return count;
}

}  // extern "C"
