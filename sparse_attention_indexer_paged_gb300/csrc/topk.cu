// Per-row top-k of the indexer logits (sparse_attn_indexer docs,
// _varlen_decode_rows: the selector keeps the k best columns of each row
// below its row end; forward_cpu: -1 pads the output; as_fp32_logits: BF16
// logits are read as their exact fp32 values).
//
// One CTA per row: 1024 threads and one row per SM, or 512 threads and two
// rows per SM where a grid has more rows than the device has SMs.  Scores map
// to order-preserving 32-bit keys (NaN lowest, -0 == +0); the k-th largest
// key tau and the number of keys equal to tau that are kept (the lowest
// columns among them) are found by radix select.
//
// Sampled path (rows up to kFastMaxCols columns), one full read of the row:
//   sample  every sv-th 4-column group (at most kSampleQuads groups); the
//           sample's ks-th largest key (ks ~ 1.5 k / sv, two radix rounds),
//           cut to its top 22 bits, is a threshold t;
//   pass    scores at or above t's float form go to per-warp candidate
//           slices (a ballot per key position, the count in a register),
//           packed afterwards;
//   then    if at least k and at most kCandCap keys reached t, tau is found
//           on the candidates alone (all keys >= tau are among them; radix
//           digits start at their highest differing bit), the kept
//           candidates set their bits in two shared-memory bitmaps and one
//           block-wide scan over the bitmaps writes the chosen columns in
//           ascending order.
// Otherwise (the sample missed, or the row is longer) the exact passes run:
// a histogram of the top 11 key bits, then either the bitmap/candidate pass
// above on that bin's keys, or two more histogram passes and an ordered
// compaction of the row.
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kBins = 2048;
constexpr int kPerThread = 8;          // elements per thread per chunk of the ordered pass
constexpr int kLoadsInFlight = 4;      // 16-byte loads per thread per iteration
// 4-column groups in the threshold sample: 4096 keys (a 16384-key sample
// measured ~3 us slower per launch)
constexpr int kSampleQuads = 1024;

// Geometry of the long-row kernel: kT threads; two shared-memory bitmaps
// over kMaxCols columns; kCap (key, column) candidates; kMinBlocks CTAs an SM
// must hold.  The stage area takes the threshold sample's keys, then the
// warps' candidate columns.
template <int kT, int kMaxCols, int kCap, int kMinBlocks_>
struct TopkCfg {
  static constexpr int kThreads = kT;
  static constexpr int kWarps = kT / 32;
  static constexpr int kMinBlocks = kMinBlocks_;
  static constexpr int kFastMaxCols = kMaxCols;
  static constexpr int kBitmapWords = kMaxCols / 32;
  static constexpr int kCandCap = kCap;
  static constexpr int kStageBytes = kSampleQuads * 16 > kCap * 4 ? kSampleQuads * 16 : kCap * 4;
  // dynamic shared memory map
  static constexpr int kOffHist = 0;                              // uint32 [kBins]
  static constexpr int kOffSel = kOffHist + kBins * 4;            // uint32 [kBitmapWords]
  static constexpr int kOffTie = kOffSel + kBitmapWords * 4;      // uint32 [kBitmapWords]
  static constexpr int kOffCandKey = kOffTie + kBitmapWords * 4;  // uint32 [kCandCap]
  static constexpr int kOffCandCol = kOffCandKey + kCandCap * 4;  // int32  [kCandCap]
  static constexpr int kOffStage = kOffCandCol + kCandCap * 4;
  static constexpr int kSmemBytes = kOffStage + kStageBytes;
  static_assert(kBins % kT == 0 && kT <= 1024, "each thread owns a whole number of histogram bins");
  static_assert(kCap % (32 * kWarps) == 0, "whole warp slices of candidates");
  static_assert(kSmemBytes * kMinBlocks <= 232448 - 1024 * (kMinBlocks - 1), "over the shared memory of an SM");
};
// one row per SM, rows up to 2^18 columns on the sampled path
using WideCfg = TopkCfg<1024, 1 << 18, 8192, 1>;
// two rows per SM (grids of more rows than SMs), rows up to 2^17 columns
using HalfCfg = TopkCfg<512, 1 << 17, 6144, 2>;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below every number
  if (u == 0x80000000u) u = 0u;                     // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The smallest score whose key reaches t (t >= 1): for every non-NaN score x,
// order_key(x) >= t exactly when x >= key_floor(t).  NaN scores fail the
// comparison, as their key 0 fails t >= 1; a t above the key of +inf gives
// NaN, which no score reaches.
__device__ __forceinline__ float key_floor(uint32_t t) {
  if (t & 0x80000000u) return __uint_as_float(t & 0x7fffffffu);
  const uint32_t u = ~t;  // a negative score's key is its complemented bits
  return u > 0xff800000u ? -INFINITY : __uint_as_float(u);
}

template <typename LT>
__device__ __forceinline__ float load_score(const LT* row, int64_t i);
template <>
__device__ __forceinline__ float load_score<float>(const float* row, int64_t i) {
  return row[i];
}
template <>
__device__ __forceinline__ float load_score<__nv_bfloat16>(const __nv_bfloat16* row, int64_t i) {
  return __bfloat162float(row[i]);
}

// Four consecutive scores starting at a multiple of 4, as a raw vector.
template <typename LT> struct Vec4;
template <> struct Vec4<float> {
  using T = float4;
  __device__ static T load(const float* row, int64_t i) {
    return __ldg(reinterpret_cast<const float4*>(row + i));
  }
  __device__ static void keys(const T& v, uint32_t (&k)[4]) {
    k[0] = order_key(v.x);
    k[1] = order_key(v.y);
    k[2] = order_key(v.z);
    k[3] = order_key(v.w);
  }
  __device__ static void vals(const T& v, float (&x)[4]) {
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
};
template <> struct Vec4<__nv_bfloat16> {
  using T = uint2;
  __device__ static T load(const __nv_bfloat16* row, int64_t i) {
    return __ldg(reinterpret_cast<const uint2*>(row + i));
  }
  __device__ static void keys(const T& v, uint32_t (&k)[4]) {
    k[0] = order_key(__uint_as_float(v.x << 16));
    k[1] = order_key(__uint_as_float(v.x & 0xffff0000u));
    k[2] = order_key(__uint_as_float(v.y << 16));
    k[3] = order_key(__uint_as_float(v.y & 0xffff0000u));
  }
  __device__ static void vals(const T& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};

__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix sum of 32-bit values over a block of kT threads; *total =
// block sum.
template <int kT>
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t v, uint32_t* buf, uint32_t* total) {
  constexpr int kWarps = kT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t inc = warp_incl_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = warp_incl_sum(lane < kWarps ? buf[lane] : 0u);
    if (lane < kWarps) buf[lane] = x;
  }
  __syncthreads();
  const uint32_t before = warp ? buf[warp - 1] : 0u;
  *total = buf[kWarps - 1];
  __syncthreads();
  return before + inc - v;
}

// Walk the row [a, b) in 4-column groups with kLoadsInFlight loads per thread
// in flight; fn(first column, keys[4], valid mask) for every group.
template <int kThreads, typename LT, typename F>
__device__ __forceinline__ void for_each_quad(const LT* rp, int64_t a, int64_t b, F&& fn) {
  const int64_t a4 = a & ~static_cast<int64_t>(3);
  constexpr int64_t kStep = 4 * static_cast<int64_t>(kThreads) * kLoadsInFlight;
  for (int64_t base = a4; base < b; base += kStep) {
    typename Vec4<LT>::T v[kLoadsInFlight];
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) {
      const int64_t i = base + 4 * (threadIdx.x + static_cast<int64_t>(u) * kThreads);
      if (i + 3 < b && i >= a) v[u] = Vec4<LT>::load(rp, i);
    }
#pragma unroll
    for (int u = 0; u < kLoadsInFlight; ++u) {
      const int64_t i = base + 4 * (threadIdx.x + static_cast<int64_t>(u) * kThreads);
      if (i >= b) continue;
      uint32_t k[4];
      uint32_t valid = 0xfu;
      if (i + 3 < b && i >= a) {
        Vec4<LT>::keys(v[u], k);
      } else {
        valid = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t c = i + e;
          k[e] = 0;
          if (c >= a && c < b) {
            k[e] = order_key(load_score<LT>(rp, c));
            valid |= 1u << e;
          }
        }
      }
      fn(i, k, valid);
    }
  }
}

// Finds the bin holding the `remaining`-th largest key among the histogram's
// nbins bins (thread t of kT owns the kBins / kT bins below nbins - kPer t,
// highest first).  Returns the bin and, in *above, the number of keys in
// higher bins.
template <int kT>
__device__ __forceinline__ uint32_t find_bin(const uint32_t* hist, uint32_t nbins,
                                             uint32_t remaining, uint32_t* scan_buf,
                                             uint32_t* s_bin, uint32_t* s_above,
                                             uint32_t* above) {
  constexpr int kPer = kBins / kT;
  const int hi = static_cast<int>(nbins) - 1 - kPer * static_cast<int>(threadIdx.x);
  uint32_t h[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    h[e] = hi - e >= 0 ? hist[hi - e] : 0u;
    sum += h[e];
  }
  uint32_t tot;
  uint32_t run = block_excl_sum<kT>(sum, scan_buf, &tot);
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    if (hi - e >= 0 && run < remaining && run + h[e] >= remaining) {
      *s_bin = static_cast<uint32_t>(hi - e);
      *s_above = run;
    }
    run += h[e];
  }
  __syncthreads();
  const uint32_t bin = *s_bin;
  *above = *s_above;
  __syncthreads();
  return bin;
}

// Exact selection among the shared-memory candidates (every key of the row
// that can be in its top-k is among them, and all of them share the key bits
// above those the earlier passes left open), then the ordered output.  The
// `remaining`-th largest candidate is found by radix select over digits of
// up to 11 bits, starting at the highest bit where the candidates' largest
// and smallest keys differ and stopping once the chosen bin is taken whole
// (the candidates are the top few percent of the row and would crowd into
// one or two bins of a fixed top digit).  Chosen candidates above the last
// digit's bin, or in it when it is taken whole, set their column's bit in
// `sel`; otherwise the first take_eq keys equal to tau (lowest columns) come
// from `tie`.  A block-wide scan over the bitmaps writes the columns in
// ascending order.  sel/tie must be zero for the words [0, nwords) except
// for columns already chosen by the caller (set in sel).
template <int kThreads>
__device__ __forceinline__ void select_candidates_and_write(
    const uint32_t* cand_key, const int32_t* cand_col, int nc, uint32_t* sel, uint32_t* tie,
    int nwords, int64_t wa, uint32_t remaining, uint32_t* hist, uint32_t* scan_buf, uint32_t* s_bin,
    uint32_t* s_above, uint32_t* s_max, uint32_t* s_min, int32_t* op) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t mx = 0, mn = 0xffffffffu;
  for (int i = tid; i < nc; i += kThreads) {
    const uint32_t key = cand_key[i];
    mx = max(mx, key);
    mn = min(mn, key);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (tid == 0) {
    *s_max = 0;
    *s_min = 0xffffffffu;
  }
  __syncthreads();
  if (lane == 0) {
    atomicMax(s_max, mx);
    atomicMin(s_min, mn);
  }
  __syncthreads();
  const uint32_t kmax = *s_max;
  const uint32_t diff = kmax ^ *s_min;
  uint32_t prefix = kmax;  // all candidates equal: tau is their key
  bool whole = false;      // the last bin is taken whole: keys >= prefix are the chosen ones
  if (diff != 0) {
    int top = 31 - __clz(diff);
    uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
    prefix = kmax & mask;
#pragma unroll 1
    while (top >= 0) {
      const int lo = max(top - 10, 0);
      const uint32_t nbins = 1u << (top - lo + 1);
      for (int i = tid; i < static_cast<int>(nbins); i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < nc; i += kThreads) {
        const uint32_t key = cand_key[i];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> lo) & (nbins - 1)], 1u);
      }
      __syncthreads();
      uint32_t above;
      const uint32_t bin = find_bin<kThreads>(hist, nbins, remaining, scan_buf, s_bin, s_above, &above);
      const uint32_t cnt = hist[bin];
      __syncthreads();  // hist is cleared by the next digit
      prefix |= bin << lo;
      mask |= (nbins - 1) << lo;
      remaining -= above;
      if (cnt == remaining) {
        whole = true;
        break;
      }
      top = lo - 1;
    }
  }
  const uint32_t tau = prefix;
  const uint32_t take_eq = whole ? 0u : remaining;
  for (int i = tid; i < nc; i += kThreads) {
    const uint32_t key = cand_key[i];
    const int64_t off = cand_col[i] - wa;
    if (whole ? key >= tau : key > tau) atomicOr(&sel[off >> 5], 1u << (off & 31));
    else if (key == tau) atomicOr(&tie[off >> 5], 1u << (off & 31));
  }
  __syncthreads();
  const int per = (nwords + kThreads - 1) / kThreads;
  const int w0 = tid * per, w1 = min(nwords, w0 + per);
  uint32_t nsel = 0, ntie = 0;
  for (int w = w0; w < w1; ++w) {
    nsel += __popc(sel[w]);
    ntie += __popc(tie[w]);
  }
  uint32_t tot;
  const uint32_t ex = block_excl_sum<kThreads>(nsel | (ntie << 16), scan_buf, &tot);
  uint32_t sel_before = ex & 0xffffu, tie_before = ex >> 16;
  for (int w = w0; w < w1; ++w) {
    uint32_t ms = sel[w], mt = tie[w];
    while (ms | mt) {
      const uint32_t m = ms | mt;
      const int bit = __ffs(m) - 1;
      const int32_t col = static_cast<int32_t>(wa + 32 * static_cast<int64_t>(w) + bit);
      if ((ms >> bit) & 1u) {
        op[sel_before + min(tie_before, take_eq)] = col;
        ++sel_before;
      } else {
        if (tie_before < take_eq) op[sel_before + tie_before] = col;
        ++tie_before;
      }
      ms &= ~(1u << bit);
      mt &= ~(1u << bit);
    }
  }
}

template <typename LT, typename C>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks)
    topk_kernel(const LT* __restrict__ logits, int64_t stride, const int32_t* __restrict__ starts,
                const int32_t* __restrict__ ends, int32_t k, int32_t* __restrict__ out,
                int64_t out_stride, int32_t* status) {
  grid_dep_wait();  // the logits come from the kernel before this one
  constexpr int kThreads = C::kThreads, kWarps = C::kWarps;
  constexpr int kFastMaxCols = C::kFastMaxCols, kCandCap = C::kCandCap;
  constexpr int kOffHist = C::kOffHist, kOffSel = C::kOffSel, kOffTie = C::kOffTie;
  constexpr int kOffCandKey = C::kOffCandKey, kOffCandCol = C::kOffCandCol, kOffStage = C::kOffStage;
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
  uint32_t* sel = reinterpret_cast<uint32_t*>(smem + kOffSel);
  uint32_t* tie = reinterpret_cast<uint32_t*>(smem + kOffTie);
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(smem + kOffCandKey);
  int32_t* cand_col = reinterpret_cast<int32_t*>(smem + kOffCandCol);
  __shared__ uint32_t scan_buf[kWarps];
  __shared__ uint32_t s_bin, s_above, s_ncand, s_max, s_min;
  __shared__ uint32_t s_wcount[kWarps];

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const LT* rp = logits + static_cast<int64_t>(row) * stride;
  int32_t* op = out + static_cast<int64_t>(row) * out_stride;
  const int64_t a = starts ? max(starts[row], 0) : 0;
  const int64_t b = min(static_cast<int64_t>(ends[row]), stride);
  const int64_t len = b > a ? b - a : 0;

  if (len <= k) {  // every column is chosen, then -1
    for (int64_t i = tid; i < k; i += kThreads) op[i] = i < len ? static_cast<int32_t>(a + i) : -1;
    return;
  }

  const int64_t wa = a & ~static_cast<int64_t>(31);
  const int nwords = static_cast<int>((b - wa + 31) >> 5);
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t above;
  // the sampled path reads whole 4-column groups as one vector load (16
  // bytes of fp32, 8 of bf16): every row must start on a 16-byte boundary
  if (b - wa <= kFastMaxCols && stride % (16 / static_cast<int64_t>(sizeof(LT))) == 0) {
    // ---- sampled threshold: every sv-th 4-column group, at most kSampleQuads
    // groups; the sample's ks-th largest key, rounded down to its top 22
    // bits, is a threshold t that about 1.5 k keys of the row reach
    const int64_t a4 = a & ~static_cast<int64_t>(3);
    const int64_t nquads = (b - a4 + 3) >> 2;
    const int64_t sv = (nquads + kSampleQuads - 1) / kSampleQuads;
    const int nsq = static_cast<int>((nquads + sv - 1) / sv);
    uint32_t* skey = reinterpret_cast<uint32_t*>(smem + kOffStage);
    for (int q = tid; q < nsq; q += kThreads) {
      const int64_t i = a4 + 4 * (static_cast<int64_t>(q) * sv);
      uint32_t kq[4];
      if (i >= a && i + 3 < b) {
        Vec4<LT>::keys(Vec4<LT>::load(rp, i), kq);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) kq[e] = (i + e >= a && i + e < b) ? order_key(load_score<LT>(rp, i + e)) : 0u;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) skey[4 * q + e] = kq[e];  // out-of-row columns: key 0, the lowest
    }
    for (int i = tid; i < nwords; i += kThreads) {
      sel[i] = 0;
      tie[i] = 0;
    }
    if (tid < kWarps) s_wcount[tid] = 0;
    const int ns = 4 * nsq;
    const int64_t want = sv == 1 ? k : (3 * static_cast<int64_t>(k)) / (2 * sv) + 16;
    uint32_t t = 0;  // stays 0 if the sample is not larger than want: every non-NaN score qualifies
    if (want < ns) {
      uint32_t prefix = 0, prefix_mask = 0, remaining = static_cast<uint32_t>(want);
#pragma unroll 1
      for (int round = 0; round < 2; ++round) {
        const int shift = round == 0 ? 21 : 10;
        for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < ns; i += kThreads) {
          const uint32_t key = skey[i];
          if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> shift) & 2047u], 1u);
        }
        __syncthreads();
        const uint32_t bin = find_bin<kThreads>(hist, 2048, remaining, scan_buf, &s_bin, &s_above, &above);
        prefix |= bin << shift;
        prefix_mask |= 2047u << shift;
        remaining -= above;
      }
      t = prefix;
    }
    __syncthreads();
    // ---- one pass over the row: keys >= t become candidates.  The scores
    // are compared with t's float form; only candidates are turned into keys.
    // t >= 1 leaves out NaN scores (key 0): if fewer than k keys then reach
    // t, the exact passes below run.  Each warp appends to its own slice of
    // the candidate arrays; about 1.5 k of the row's scores reach t, so a
    // 4-score vector is tested by its maximum first and a candidate takes its
    // slot with one shared atomic on the warp's counter (the counter keeps
    // counting past the slice, which marks an overflow); the slices are
    // packed afterwards.
    t = max(t, 1u);
    const float tf = key_floor(t);
    constexpr int kWarpCap = kCandCap / kWarps;
    uint32_t* wkey = cand_key + warp * kWarpCap;  // this warp's slice, packed later
    int32_t* wcol = reinterpret_cast<int32_t*>(smem + kOffStage) + warp * kWarpCap;
    uint32_t* wcnt = s_wcount + warp;
    // columns as 32-bit offsets from a4 (rows are far below 2^31 columns),
    // eight 16-byte loads a thread in flight
    constexpr int kPassLoads = 8;
    constexpr int32_t kStep = 4 * kThreads * kPassLoads;
    const LT* rq = rp + a4;
    const int32_t na = static_cast<int32_t>(a - a4), nb = static_cast<int32_t>(b - a4);
    const int32_t col0 = static_cast<int32_t>(a4);
    for (int32_t base = 0; base < nb; base += kStep) {
      typename Vec4<LT>::T v[kPassLoads];
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        const int32_t i = base + 4 * (tid + u * kThreads);
        if (i + 3 < nb && i >= na) v[u] = Vec4<LT>::load(rq, i);
      }
#pragma unroll
      for (int u = 0; u < kPassLoads; ++u) {
        const int32_t i = base + 4 * (tid + u * kThreads);
        float xq[4];
        if (i + 3 < nb && i >= na) {
          Vec4<LT>::vals(v[u], xq);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) xq[e] = (i + e >= na && i + e < nb) ? load_score<LT>(rq, i + e) : __int_as_float(0x7fffffff);
        }
        // fmaxf ignores a NaN operand; an all-NaN vector has no candidate
        if (fmaxf(fmaxf(xq[0], xq[1]), fmaxf(xq[2], xq[3])) >= tf) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (xq[e] >= tf) {
              const uint32_t slot = atomicAdd(wcnt, 1u);
              if (slot < static_cast<uint32_t>(kWarpCap)) {
                wkey[slot] = order_key(xq[e]);
                wcol[slot] = col0 + i + e;
              }
            }
          }
        }
      }
    }
    __syncthreads();
    // pack the slices: cand_key in place (slices only move down), columns
    // from the ring area into cand_col
    {
      const uint32_t cnt = lane < kWarps ? min(s_wcount[lane], static_cast<uint32_t>(kWarpCap)) : 0u;
      bool over = false;
      uint32_t before = 0, total = 0;
      // every warp computes the exclusive prefix of the 32 slice counts
      const uint32_t inc = warp_incl_sum(cnt);
      before = inc - cnt;
      total = __shfl_sync(0xffffffffu, inc, 31);
      over = __any_sync(0xffffffffu, lane < kWarps && s_wcount[lane] > static_cast<uint32_t>(kWarpCap));
      const uint32_t my_before = __shfl_sync(0xffffffffu, before, warp);
      const uint32_t my_cnt = __shfl_sync(0xffffffffu, cnt, warp);
      uint32_t keys_tmp[kWarpCap / 32];
      int32_t cols_tmp[kWarpCap / 32];
#pragma unroll
      for (int r = 0; r < kWarpCap / 32; ++r) {
        const uint32_t j = static_cast<uint32_t>(r * 32 + lane);
        if (j < my_cnt) {
          keys_tmp[r] = wkey[j];
          cols_tmp[r] = wcol[j];
        }
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kWarpCap / 32; ++r) {
        const uint32_t j = static_cast<uint32_t>(r * 32 + lane);
        if (j < my_cnt) {
          cand_key[my_before + j] = keys_tmp[r];
          cand_col[my_before + j] = cols_tmp[r];
        }
      }
      if (tid == 0) s_ncand = over ? 0xffffffffu : total;
    }
    __syncthreads();
    const uint32_t nc = s_ncand;
    if (nc >= static_cast<uint32_t>(k) && nc <= static_cast<uint32_t>(kCandCap)) {
      select_candidates_and_write<kThreads>(cand_key, cand_col, static_cast<int>(nc), sel, tie, nwords, wa,
                                            static_cast<uint32_t>(k), hist, scan_buf, &s_bin, &s_above, &s_max,
                                            &s_min, op);
      return;
    }
    __syncthreads();  // the sample missed (rare): exact passes below
  }

  // ---- pass 1: top 11 key bits
  for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
  __syncthreads();
  for_each_quad<kThreads, LT>(rp, a, b, [&](int64_t, const uint32_t (&kq)[4], uint32_t valid) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((valid >> e) & 1u) atomicAdd(&hist[kq[e] >> 21], 1u);
  });
  __syncthreads();
  const uint32_t b1 = find_bin<kThreads>(hist, 2048, static_cast<uint32_t>(k), scan_buf, &s_bin, &s_above, &above);
  uint32_t remaining = static_cast<uint32_t>(k) - above;
  const uint32_t c1 = hist[b1];
  __syncthreads();

  const bool fast = (b - wa) <= kFastMaxCols && c1 <= static_cast<uint32_t>(kCandCap);
  if (fast) {
    for (int i = tid; i < nwords; i += kThreads) {
      sel[i] = 0;
      tie[i] = 0;
    }
    if (tid == 0) s_ncand = 0;
    __syncthreads();
    // ---- pass 2: mark keys above the bin, collect the bin's candidates
    for_each_quad<kThreads, LT>(rp, a, b, [&](int64_t i, const uint32_t (&kq)[4], uint32_t valid) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!((valid >> e) & 1u)) continue;
        const uint32_t d = kq[e] >> 21;
        const int64_t off = i + e - wa;
        if (d > b1) {
          atomicOr(&sel[off >> 5], 1u << (off & 31));
        } else if (d == b1) {
          const uint32_t slot = atomicAdd(&s_ncand, 1u);
          if (slot < static_cast<uint32_t>(kCandCap)) {  // always: the bin holds c1 <= kCandCap keys
            cand_key[slot] = kq[e];
            cand_col[slot] = static_cast<int32_t>(i + e);
          }
        }
      }
    });
    __syncthreads();
    const int nc = min(static_cast<int>(s_ncand), kCandCap);
    select_candidates_and_write<kThreads>(cand_key, cand_col, nc, sel, tie, nwords, wa, remaining, hist, scan_buf,
                                          &s_bin, &s_above, &s_max, &s_min, op);
    return;
  }

  // ---- general path: remaining two digits over the whole row, then an
  // ordered compaction of the row.
  uint32_t prefix = b1 << 21, prefix_mask = 0x7ffu << 21;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t nbins = pass == 0 ? 2048u : 1024u;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for_each_quad<kThreads, LT>(rp, a, b, [&](int64_t, const uint32_t (&kq)[4], uint32_t valid) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (((valid >> e) & 1u) && (kq[e] & prefix_mask) == prefix)
          atomicAdd(&hist[(kq[e] >> shift) & (nbins - 1)], 1u);
    });
    __syncthreads();
    const uint32_t bin = find_bin<kThreads>(hist, nbins, remaining, scan_buf, &s_bin, &s_above, &above);
    prefix |= bin << shift;
    prefix_mask |= (nbins - 1) << shift;
    remaining -= above;
  }
  const uint32_t tau = prefix;
  const uint32_t take_eq = remaining;
  uint32_t gt_run = 0, eq_run = 0;
  for (int64_t base = a; base < b; base += static_cast<int64_t>(kThreads) * kPerThread) {
    const int64_t c0 = base + static_cast<int64_t>(tid) * kPerThread;
    uint32_t gt_bits = 0, eq_bits = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int64_t c = c0 + e;
      if (c < b) {
        const uint32_t key = order_key(load_score<LT>(rp, c));
        gt_bits |= (key > tau ? 1u : 0u) << e;
        eq_bits |= (key == tau ? 1u : 0u) << e;
      }
    }
    const uint32_t packed =
        static_cast<uint32_t>(__popc(gt_bits)) | (static_cast<uint32_t>(__popc(eq_bits)) << 16);
    uint32_t tot;
    const uint32_t ex = block_excl_sum<kThreads>(packed, scan_buf, &tot);
    uint32_t gt_before = gt_run + (ex & 0xffffu);
    uint32_t eq_before = eq_run + (ex >> 16);
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      if ((gt_bits >> e) & 1u) {
        op[gt_before + min(eq_before, take_eq)] = static_cast<int32_t>(c0 + e);
        ++gt_before;
      } else if ((eq_bits >> e) & 1u) {
        if (eq_before < take_eq) op[gt_before + eq_before] = static_cast<int32_t>(c0 + e);
        ++eq_before;
      }
    }
    gt_run += tot & 0xffffu;
    eq_run += tot >> 16;
  }
}

// ---------------------------------------------------------------------------
// Short rows (every row fits in kCols columns: the row stride is at most
// kCols).  The row's keys stay in shared memory.  An exact radix select over
// digits of up to 11 bits, starting at the highest bit where the row's keys
// differ and stopping once the chosen bin is taken whole, finds the k-th
// largest key tau; one ordered ballot pass over the row then writes the
// columns above tau and the lowest columns equal to tau, ascending.  512
// threads and kCols * 4 + 8 KB of shared memory let several rows share an
// SM, where the long-row kernel keeps one.
constexpr int kShortThreads = 512;
constexpr int kShortWarps = kShortThreads / 32;
template <int kCols> constexpr int kShortSmem = kCols * 4 + kBins * 4;

__device__ __forceinline__ uint32_t short_excl_sum(uint32_t v, uint32_t* buf, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t inc = warp_incl_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t s = warp_incl_sum(lane < kShortWarps ? buf[lane] : 0u);
    if (lane < kShortWarps) buf[lane] = s;
  }
  __syncthreads();
  const uint32_t before = warp ? buf[warp - 1] : 0u;
  *total = buf[kShortWarps - 1];
  __syncthreads();
  return before + inc - v;
}

template <typename LT, int kCols>
__global__ void __launch_bounds__(kShortThreads, kCols <= 8192 ? 4 : 3)
    topk_short_kernel(const LT* __restrict__ logits, int64_t stride, const int32_t* __restrict__ starts,
                      const int32_t* __restrict__ ends, int32_t k, int32_t* __restrict__ out,
                      int64_t out_stride) {
  grid_dep_wait();  // the logits come from the kernel before this one
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);  // [kCols], column a + i at i
  uint32_t* hist = keys + kCols;                       // [kBins]
  __shared__ uint32_t scan_buf[kShortWarps];
  __shared__ uint32_t s_max, s_min, s_bin, s_above, s_cnt;
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const LT* rp = logits + static_cast<int64_t>(row) * stride;
  int32_t* op = out + static_cast<int64_t>(row) * out_stride;
  const int64_t a = starts ? max(starts[row], 0) : 0;
  const int64_t b = min(static_cast<int64_t>(ends[row]), stride);
  const int n = b > a ? static_cast<int>(b - a) : 0;  // <= stride <= kCols
  if (n <= k) {
    for (int i = tid; i < k; i += kShortThreads) op[i] = i < n ? static_cast<int32_t>(a + i) : -1;
    return;
  }
  constexpr int kQuads = kCols / 4 / kShortThreads;  // 4-column groups a thread covers
  static_assert(kQuads % 4 == 0, "quads come in batches of 4");
  uint4* keys4 = reinterpret_cast<uint4*>(keys);
  if (tid == 0) {
    s_max = 0;
    s_min = 0xffffffffu;
  }
  // 1. the row's keys, their largest and smallest: the keys all share the
  // bits above the highest bit where the largest and smallest differ
  uint32_t mx = 0, mn = 0xffffffffu;
  if ((a & 3) == 0) {  // 16-byte (bf16: 8-byte) aligned groups of 4 columns, 4 loads in flight
#pragma unroll
    for (int u0 = 0; u0 < kQuads; u0 += 4) {
      typename Vec4<LT>::T v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = 4 * (tid + (u0 + u) * kShortThreads);
        if (i + 3 < n) v[u] = Vec4<LT>::load(rp, a + i);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int q = tid + (u0 + u) * kShortThreads, i = 4 * q;
        if (i >= n) continue;
        uint32_t kq[4];
        if (i + 3 < n) {
          Vec4<LT>::keys(v[u], kq);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) kq[e] = i + e < n ? order_key(load_score<LT>(rp, a + i + e)) : 0u;
        }
        keys4[q] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < n) {
            mx = max(mx, kq[e]);
            mn = min(mn, kq[e]);
          }
      }
    }
  } else {
#pragma unroll 8
    for (int i = tid; i < n; i += kShortThreads) {
      const uint32_t key = order_key(load_score<LT>(rp, a + i));
      keys[i] = key;
      mx = max(mx, key);
      mn = min(mn, key);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  __syncthreads();  // s_max, s_min initialised
  if (lane == 0) {
    atomicMax(&s_max, mx);
    atomicMin(&s_min, mn);
  }
  __syncthreads();
  const uint32_t kmax = s_max;
  const uint32_t diff = kmax ^ s_min;
  // 2. the k-th largest key: digits from the highest differing bit down
  uint32_t prefix = kmax, remaining = static_cast<uint32_t>(k);
  bool whole = false;  // the last chosen bin is taken whole: keys >= prefix are exactly k
  if (diff != 0) {
    int top = 31 - __clz(diff);
    uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
    prefix = kmax & mask;
#pragma unroll 1
    while (top >= 0) {
      const int lo = max(top - 10, 0);
      const uint32_t nbins = 1u << (top - lo + 1);
      for (int i = tid; i < static_cast<int>(nbins); i += kShortThreads) hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kQuads; ++u) {
        const int q = tid + u * kShortThreads, i = 4 * q;
        if (i >= n) continue;
        const uint4 k4 = keys4[q];
        const uint32_t kq[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < n && (kq[e] & mask) == prefix) atomicAdd(&hist[(kq[e] >> lo) & (nbins - 1)], 1u);
      }
      __syncthreads();
      // thread t owns bins nbins-1-4t down to nbins-4-4t (descending order)
      const int hb = static_cast<int>(nbins) - 1 - 4 * tid;
      uint32_t h[4], sum = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = hb - e >= 0 ? hist[hb - e] : 0u;
        sum += h[e];
      }
      uint32_t tot;
      const uint32_t ab = short_excl_sum(sum, scan_buf, &tot);
      if (ab < remaining && ab + sum >= remaining) {
        uint32_t acc = ab;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (acc + h[e] >= remaining) {
            s_bin = static_cast<uint32_t>(hb - e);
            s_above = acc;
            s_cnt = h[e];
            break;
          }
          acc += h[e];
        }
      }
      __syncthreads();
      prefix |= s_bin << lo;
      mask |= (nbins - 1u) << lo;
      remaining -= s_above;
      whole = s_cnt == remaining;
      __syncthreads();
      if (whole) break;
      top = lo - 1;
    }
  }
  // now: whole -> the chosen columns are those with key >= prefix; else tau =
  // prefix, chosen = keys above tau plus the first `remaining` keys equal to it
  const uint32_t take_eq = whole ? 0u : remaining;
  // 3. ascending output: warp w walks its block of columns 32 at a time
  const int per_warp = (n + kShortThreads - 1) / kShortThreads * 32;
  const int c0 = warp * per_warp, c1 = min(c0 + per_warp, n);
  uint32_t gt_w = 0, eq_w = 0;
  for (int c = c0; c < c1; c += 32) {
    const int i = c + lane;
    const uint32_t key = i < c1 ? keys[i] : 0u;
    const bool g = i < c1 && (whole ? key >= prefix : key > prefix);
    const bool e = i < c1 && !whole && key == prefix;
    gt_w += __popc(__ballot_sync(0xffffffffu, g));
    eq_w += __popc(__ballot_sync(0xffffffffu, e));
  }
  uint32_t tot;
  const uint32_t wbase = short_excl_sum(lane == 0 ? (gt_w | (eq_w << 16)) : 0u, scan_buf, &tot);
  const uint32_t wb = __shfl_sync(0xffffffffu, wbase, 0);
  uint32_t gt_run = wb & 0xffffu, eq_run = wb >> 16;
  const uint32_t lt = (1u << lane) - 1u;
  for (int c = c0; c < c1; c += 32) {
    const int i = c + lane;
    const uint32_t key = i < c1 ? keys[i] : 0u;
    const bool g = i < c1 && (whole ? key >= prefix : key > prefix);
    const bool e = i < c1 && !whole && key == prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, g), be = __ballot_sync(0xffffffffu, e);
    const uint32_t gb = gt_run + __popc(bg & lt), eb = eq_run + __popc(be & lt);
    uint32_t pos = 0xffffffffu;
    if (g) pos = gb + min(eb, take_eq);
    else if (e && eb < take_eq) pos = gb + eb;
    if (pos < static_cast<uint32_t>(k)) op[pos] = static_cast<int32_t>(a + i);
    gt_run += __popc(bg);
    eq_run += __popc(be);
  }
}

template <typename LT, typename C>
cudaError_t launch_long(const void* logits, int64_t stride, const int32_t* starts, const int32_t* ends,
                        int32_t num_rows, int32_t k, int32_t* out, int64_t out_stride, int32_t* status,
                        cudaStream_t stream) {
  const cudaError_t e =
      cudaFuncSetAttribute(topk_kernel<LT, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(topk_kernel<LT, C>, dim3(num_rows), dim3(C::kThreads), C::kSmemBytes, stream,
                          static_cast<const LT*>(logits), stride, starts, ends, k, out, out_stride, status);
}

template <typename LT, int kCols>
cudaError_t launch_short(const void* logits, int64_t stride, const int32_t* starts, const int32_t* ends,
                         int32_t num_rows, int32_t k, int32_t* out, int64_t out_stride, cudaStream_t stream) {
  const cudaError_t e = cudaFuncSetAttribute(topk_short_kernel<LT, kCols>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kShortSmem<kCols>);
  if (e != cudaSuccess) return e;
  return launch_dependent(topk_short_kernel<LT, kCols>, dim3(num_rows), dim3(kShortThreads), kShortSmem<kCols>,
                          stream, static_cast<const LT*>(logits), stride, starts, ends, k, out, out_stride);
}

}  // namespace

cudaError_t launch_top_k(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                         const int32_t* row_starts, const int32_t* row_ends, int32_t num_rows,
                         int32_t k, int32_t* out_idx, int64_t out_stride, int32_t* status,
                         cudaStream_t stream) {
  // short rows: several rows per SM
  if (logits_stride <= 8192)
    return logits_dtype == DSA_LOGITS_BF16
               ? launch_short<__nv_bfloat16, 8192>(logits, logits_stride, row_starts, row_ends, num_rows, k, out_idx,
                                                   out_stride, stream)
               : launch_short<float, 8192>(logits, logits_stride, row_starts, row_ends, num_rows, k, out_idx,
                                           out_stride, stream);
  if (logits_stride <= 16384)
    return logits_dtype == DSA_LOGITS_BF16
               ? launch_short<__nv_bfloat16, 16384>(logits, logits_stride, row_starts, row_ends, num_rows, k,
                                                    out_idx, out_stride, stream)
               : launch_short<float, 16384>(logits, logits_stride, row_starts, row_ends, num_rows, k, out_idx,
                                            out_stride, stream);
  // long rows: one row per SM, or two where the grid has more rows than the
  // device has SMs and every row fits the half geometry
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool half = num_rows > sms && logits_stride <= HalfCfg::kFastMaxCols;
  if (logits_dtype == DSA_LOGITS_BF16)
    return half ? launch_long<__nv_bfloat16, HalfCfg>(logits, logits_stride, row_starts, row_ends, num_rows, k,
                                                      out_idx, out_stride, status, stream)
                : launch_long<__nv_bfloat16, WideCfg>(logits, logits_stride, row_starts, row_ends, num_rows, k,
                                                      out_idx, out_stride, status, stream);
  return half ? launch_long<float, HalfCfg>(logits, logits_stride, row_starts, row_ends, num_rows, k, out_idx,
                                            out_stride, status, stream)
              : launch_long<float, WideCfg>(logits, logits_stride, row_starts, row_ends, num_rows, k, out_idx,
                                            out_stride, status, stream);
}

}  // namespace dsa
