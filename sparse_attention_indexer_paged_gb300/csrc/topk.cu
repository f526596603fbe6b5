// Per-row top-k of the indexer logits (sparse_attn_indexer docs,
// _varlen_decode_rows: the selector keeps the k best columns of each row
// below its row end; forward_cpu: -1 pads the output; as_fp32_logits: BF16
// logits are read as their exact fp32 values).
//
// One CTA per row.  Scores map to order-preserving 32-bit keys (NaN lowest,
// -0 == +0).  Three histogram passes over the row (11, 11 and 10 key bits)
// find the k-th largest key tau and how many keys equal to tau are kept
// (the lowest columns among them).  A final ordered pass writes the chosen
// columns in ascending order with block-wide prefix sums.
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kPerThread = 8;  // elements per thread per chunk of the ordered pass

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below every number
  if (u == 0x80000000u) u = 0u;                     // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

// Keys of 4 consecutive columns starting at a multiple of 4.
template <typename LT>
__device__ __forceinline__ void load4_keys(const LT* row, int64_t i, uint32_t (&k)[4]);
template <>
__device__ __forceinline__ void load4_keys<float>(const float* row, int64_t i, uint32_t (&k)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(row + i);
  k[0] = order_key(v.x);
  k[1] = order_key(v.y);
  k[2] = order_key(v.z);
  k[3] = order_key(v.w);
}
template <>
__device__ __forceinline__ void load4_keys<__nv_bfloat16>(const __nv_bfloat16* row, int64_t i,
                                                          uint32_t (&k)[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(row + i);
  k[0] = order_key(__uint_as_float(v.x << 16));
  k[1] = order_key(__uint_as_float(v.x & 0xffff0000u));
  k[2] = order_key(__uint_as_float(v.y << 16));
  k[3] = order_key(__uint_as_float(v.y & 0xffff0000u));
}

__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive block prefix sum of 32-bit values; *total = block sum.
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t v, uint32_t* buf, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t inc = warp_incl_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) buf[lane] = warp_incl_sum(buf[lane]);
  __syncthreads();
  const uint32_t before = warp ? buf[warp - 1] : 0u;
  *total = buf[kWarps - 1];
  __syncthreads();
  return before + inc - v;
}

template <typename LT>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const LT* __restrict__ logits, int64_t stride, const int32_t* __restrict__ starts,
                const int32_t* __restrict__ ends, int32_t k, int32_t* __restrict__ out,
                int64_t out_stride) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t scan_buf[kWarps];
  __shared__ uint32_t s_bin, s_above;

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

  // ---- radix select of the k-th largest key
  uint32_t prefix = 0, prefix_mask = 0;
  uint32_t remaining = static_cast<uint32_t>(k);
  const int64_t a4 = a & ~static_cast<int64_t>(3);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t nbins = pass == 2 ? 1024u : 2048u;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = a4 + 4 * static_cast<int64_t>(tid); i < b; i += 4 * kThreads) {
      uint32_t kk[4];
      if (i + 3 < b && i >= a) {
        load4_keys<LT>(rp, i, kk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((kk[e] & prefix_mask) == prefix) atomicAdd(&hist[(kk[e] >> shift) & (nbins - 1)], 1u);
      } else {
        for (int e = 0; e < 4; ++e) {
          const int64_t c = i + e;
          if (c < a || c >= b) continue;
          const uint32_t key = order_key(load_score<LT>(rp, c));
          if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> shift) & (nbins - 1)], 1u);
        }
      }
    }
    __syncthreads();
    // Thread t owns bins hi = nbins-1-2t and lo = hi-1 (threads past nbins/2
    // own none); an exclusive scan gives the count of keys in higher bins.
    uint32_t h_hi = 0, h_lo = 0;
    const int hi = static_cast<int>(nbins) - 1 - 2 * tid;
    if (hi >= 1) {
      h_hi = hist[hi];
      h_lo = hist[hi - 1];
    }
    uint32_t tot;
    const uint32_t above = block_excl_sum(h_hi + h_lo, scan_buf, &tot);
    if (hi >= 1) {
      if (above < remaining && above + h_hi >= remaining) {
        s_bin = static_cast<uint32_t>(hi);
        s_above = above;
      } else if (above + h_hi < remaining && above + h_hi + h_lo >= remaining) {
        s_bin = static_cast<uint32_t>(hi - 1);
        s_above = above + h_hi;
      }
    }
    __syncthreads();
    prefix |= s_bin << shift;
    prefix_mask |= (nbins - 1) << shift;
    remaining -= s_above;
    __syncthreads();
  }
  const uint32_t tau = prefix;       // k-th largest key
  const uint32_t take_eq = remaining; // keys equal to tau that are kept (lowest columns)

  // ---- ordered compaction: column order, keys > tau, then the first take_eq ties
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
    const uint32_t packed = static_cast<uint32_t>(__popc(gt_bits)) | (static_cast<uint32_t>(__popc(eq_bits)) << 16);
    uint32_t tot;
    const uint32_t ex = block_excl_sum(packed, scan_buf, &tot);
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

}  // namespace

cudaError_t launch_top_k(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                         const int32_t* row_starts, const int32_t* row_ends, int32_t num_rows,
                         int32_t k, int32_t* out_idx, int64_t out_stride, int32_t* status,
                         cudaStream_t stream) {
  (void)status;
  if (logits_dtype == DSA_LOGITS_BF16) {
    topk_kernel<__nv_bfloat16><<<num_rows, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(logits), logits_stride, row_starts, row_ends, k, out_idx,
        out_stride);
  } else {
    topk_kernel<float><<<num_rows, kThreads, 0, stream>>>(static_cast<const float*>(logits),
                                                          logits_stride, row_starts, row_ends, k,
                                                          out_idx, out_stride);
  }
  return cudaGetLastError();
}

}  // namespace dsa
