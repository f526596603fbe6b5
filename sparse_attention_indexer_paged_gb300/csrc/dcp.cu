// Decode context parallelism (sparse_attn_indexer docs,
// _merge_dcp_topk_global): every rank scores its 1/world of each request's
// keys and takes a top-k over its shard; the ranks' candidates are packed as
// (score, global token id), all-gathered rank-major into
// [world][rows][k][2] and merged by a stable top-k into the global top-k.  A
// token in the global top-k has at most k - 1 tokens above it overall, hence
// at most k - 1 on its own rank, so it is in that rank's local top-k and the
// merge is exact.
//
// Shard mapping: keys go to ranks in blocks of `interleave` consecutive
// tokens, round robin, so local position l of rank r is global token
// ((l / I) * world + r) * I + l mod I.
//
// pack_kernel   one CTA per row: (score of the local column, global id), or
//               (-inf, -1) for a padded slot.
// merge_kernel  one CTA per row over world * k candidates: each valid one
//               becomes the 64-bit key (score key << 32) | ~global id, so keys
//               are distinct and order by larger score, then lower id; the
//               k-th largest key is found by radix select (digits of up to 11
//               bits from the highest bit where the keys differ, stopping once
//               the chosen bin is taken whole); the chosen ids are set in a
//               bitmap over the row's id range and written in ascending order
//               by one block scan, -1 padded.
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kMergeThreads = 1024;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMaxCand = DSA_DCP_MAX_WORLD * DSA_MAX_TOPK;  // 16384
constexpr int kBins = 2048;
constexpr int kChunkWords = 16384;           // id bitmap: 2^19 ids per chunk
constexpr uint32_t kChunkIds = kChunkWords * 32u;
// dynamic shared memory of the merge: keys, histogram, id bitmap
constexpr int kOffKeys = 0;
constexpr int kOffHist = kOffKeys + kMaxCand * 8;
constexpr int kOffBitmap = kOffHist + kBins * 4;
constexpr int kMergeSmem = kOffBitmap + kChunkWords * 4;
static_assert(kMergeSmem <= 232448, "over the per-CTA shared memory limit");

// Order-preserving 32-bit key of a score (the top-k kernel's order: NaN
// lowest, -0 == +0).
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename LT> __device__ __forceinline__ float load_logit(const LT* p);
template <> __device__ __forceinline__ float load_logit<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float load_logit<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

constexpr int kPackThreads = 256;
constexpr int kPackPer = 8;  // slots per thread per pass, loads issued together

template <typename LT>
__global__ void __launch_bounds__(kPackThreads)
    pack_kernel(const LT* __restrict__ logits, int64_t stride, const int32_t* __restrict__ idx,
                int64_t idx_stride, int32_t k, int32_t rank, int32_t world, int32_t inter,
                float2* __restrict__ packed) {
  const int row = blockIdx.x;
  const LT* lrow = logits + static_cast<int64_t>(row) * stride;
  const int32_t* irow = idx + static_cast<int64_t>(row) * idx_stride;
  float2* prow = packed + static_cast<int64_t>(row) * k;
  for (int base = 0; base < k; base += kPackThreads * kPackPer) {
    int32_t l[kPackPer];
    float sc[kPackPer];
#pragma unroll
    for (int u = 0; u < kPackPer; ++u) {
      const int j = base + u * kPackThreads + static_cast<int>(threadIdx.x);
      l[u] = j < k ? irow[j] : -1;
    }
#pragma unroll
    for (int u = 0; u < kPackPer; ++u) sc[u] = (l[u] >= 0 && l[u] < stride) ? load_logit<LT>(lrow + l[u]) : 0.0f;
#pragma unroll
    for (int u = 0; u < kPackPer; ++u) {
      const int j = base + u * kPackThreads + static_cast<int>(threadIdx.x);
      if (j >= k) continue;
      float2 o = make_float2(-INFINITY, -1.0f);
      if (l[u] >= 0 && l[u] < stride) {
        const int64_t g = (static_cast<int64_t>(l[u] / inter) * world + rank) * inter + l[u] % inter;
        o = make_float2(sc[u], static_cast<float>(g));
      }
      prow[j] = o;
    }
  }
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

// Exclusive block prefix sum of 32-bit values.
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t v, uint32_t* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t inc = warp_incl_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) buf[lane] = warp_incl_sum(buf[lane]);
  __syncthreads();
  const uint32_t before = warp ? buf[warp - 1] : 0u;
  __syncthreads();
  return before + inc - v;
}

// Key of a packed candidate; 0 for a padded slot.  A valid key is never 0:
// its low word is ~gid and gid < 2^24.
__device__ __forceinline__ uint64_t cand_key(float2 c) {
  if (!(c.y >= 0.0f)) return 0;
  const uint32_t gid = static_cast<uint32_t>(c.y);
  return (static_cast<uint64_t>(score_key(c.x)) << 32) | static_cast<uint32_t>(~gid);
}
__device__ __forceinline__ int32_t key_gid(uint64_t key) {
  return static_cast<int32_t>(~static_cast<uint32_t>(key));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(0xffffffffu, x, o);
    x = y > x ? y : x;
  }
  return x;
}

constexpr int kLoadPer = kMaxCand / kMergeThreads;  // 16 slots per thread
constexpr int kSlotsPerRank = DSA_MAX_TOPK / kMergeThreads;
static_assert(kLoadPer == DSA_DCP_MAX_WORLD * kSlotsPerRank, "slot split");
static_assert(kChunkWords == kMergeThreads * 16, "bitmap scan: 16 words per thread");

__global__ void __launch_bounds__(kMergeThreads, 1)
    merge_kernel(const float2* __restrict__ gathered, int32_t world, int32_t rows, int32_t k,
                 int32_t* __restrict__ out, int64_t out_stride) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem + kOffKeys);  // slot r * k + j
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + kOffBitmap);
  __shared__ uint32_t scan_buf[kMergeWarps];
  __shared__ unsigned long long s_max, s_or;
  __shared__ uint32_t s_nv, s_maxgid, s_bin, s_above, s_cnt;
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int n = world * k;
  if (tid == 0) {
    s_nv = 0;
    s_maxgid = 0;
    s_max = 0;
    s_or = 0;
  }
  __syncthreads();

  // 1. every slot's key; a thread's loads are issued together
  {
    float2 v[kLoadPer];
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_WORLD; ++r)
#pragma unroll
      for (int h = 0; h < kSlotsPerRank; ++h) {
        const int j = h * kMergeThreads + tid;
        v[r * kSlotsPerRank + h] = (r < world && j < k)
                                       ? gathered[(static_cast<int64_t>(r) * rows + row) * k + j]
                                       : make_float2(0.0f, -1.0f);
      }
    uint32_t nv = 0, mg = 0;
    uint64_t mx = 0;
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_WORLD; ++r)
#pragma unroll
      for (int h = 0; h < kSlotsPerRank; ++h) {
        const int j = h * kMergeThreads + tid;
        const uint64_t key = cand_key(v[r * kSlotsPerRank + h]);
        if (r < world && j < k) keys[r * k + j] = key;
        if (key != 0) {
          ++nv;
          mg = max(mg, static_cast<uint32_t>(key_gid(key)));
          mx = key > mx ? key : mx;
        }
      }
    nv = __reduce_add_sync(0xffffffffu, nv);
    mg = __reduce_max_sync(0xffffffffu, mg);
    mx = warp_max_u64(mx);
    if (lane == 0) {
      atomicAdd(&s_nv, nv);
      atomicMax(&s_maxgid, mg);
      atomicMax(&s_max, static_cast<unsigned long long>(mx));
    }
  }
  __syncthreads();
  const int nv = static_cast<int>(s_nv);
  const int take = min(nv, k);
  const uint64_t kmax = s_max;

  // 2. the highest bit where valid keys differ
  {
    uint64_t x = 0;
#pragma unroll 4
    for (int u = 0; u < kLoadPer; ++u) {
      const int i = u * kMergeThreads + tid;
      if (i >= n) break;
      const uint64_t key = keys[i];
      if (key != 0) x |= key ^ kmax;
    }
    const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(x >> 32));
    const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(x));
    if (lane == 0 && (hi | lo)) atomicOr(&s_or, (static_cast<unsigned long long>(hi) << 32) | lo);
  }
  __syncthreads();
  const uint64_t diff = s_or;

  // 3. the take-th largest key, digits of up to 11 bits from the highest
  // differing bit down; stop once the chosen bin is taken whole
  uint64_t tau = 1;  // all valid keys
  if (take > 0 && take < nv) {
    int top = 63 - __clzll(static_cast<long long>(diff));  // take < nv: at least two distinct keys
    uint64_t mask = top >= 63 ? 0 : ~((uint64_t{1} << (top + 1)) - 1);
    uint64_t prefix = kmax & mask;
    uint32_t remaining = static_cast<uint32_t>(take);
#pragma unroll 1
    while (top >= 0) {
      const int lo = max(top - 10, 0);
      const uint32_t nbins = 1u << (top - lo + 1);
      for (int i = tid; i < static_cast<int>(nbins); i += kMergeThreads) hist[i] = 0;
      __syncthreads();
#pragma unroll 4
      for (int u = 0; u < kLoadPer; ++u) {
        const int i = u * kMergeThreads + tid;
        if (i >= n) break;
        const uint64_t key = keys[i];
        if (key != 0 && (key & mask) == prefix) atomicAdd(&hist[(key >> lo) & (nbins - 1)], 1u);
      }
      __syncthreads();
      // thread t owns bins nbins-1-2t and nbins-2-2t (descending order)
      const int hb = static_cast<int>(nbins) - 1 - 2 * tid;
      uint32_t h_hi = 0, h_lo = 0;
      if (hb >= 1) {
        h_hi = hist[hb];
        h_lo = hist[hb - 1];
      }
      const uint32_t ab = block_excl_sum(h_hi + h_lo, scan_buf);
      if (hb >= 1) {
        if (ab < remaining && ab + h_hi >= remaining) {
          s_bin = static_cast<uint32_t>(hb);
          s_above = ab;
          s_cnt = h_hi;
        } else if (ab + h_hi < remaining && ab + h_hi + h_lo >= remaining) {
          s_bin = static_cast<uint32_t>(hb - 1);
          s_above = ab + h_hi;
          s_cnt = h_lo;
        }
      }
      __syncthreads();
      prefix |= static_cast<uint64_t>(s_bin) << lo;
      mask |= static_cast<uint64_t>(nbins - 1) << lo;
      remaining -= s_above;
      const bool whole = s_cnt == remaining;
      __syncthreads();
      if (whole) break;  // every key with this prefix is taken: keys >= prefix are exactly `take`
      top = lo - 1;
    }
    tau = prefix;
  }

  // 4. the chosen ids in ascending order: a bitmap over the row's id range,
  // 2^19 ids at a time, scanned in order (16 words per thread)
  int32_t* orow = out + static_cast<int64_t>(row) * out_stride;
  uint32_t written = 0;
  const uint32_t maxgid = s_maxgid;
  for (uint32_t c0 = 0; take > 0 && c0 <= maxgid; c0 += kChunkIds) {
    uint4* bm4 = reinterpret_cast<uint4*>(bitmap);
#pragma unroll
    for (int u = 0; u < kChunkWords / 4 / kMergeThreads; ++u) bm4[u * kMergeThreads + tid] = make_uint4(0, 0, 0, 0);
    __syncthreads();
#pragma unroll 4
    for (int u = 0; u < kLoadPer; ++u) {
      const int i = u * kMergeThreads + tid;
      if (i >= n) break;
      const uint64_t key = keys[i];
      const uint32_t off = static_cast<uint32_t>(key_gid(key)) - c0;
      if (key != 0 && key >= tau && off < kChunkIds) atomicOr(&bitmap[off >> 5], 1u << (off & 31));
    }
    __syncthreads();
    uint4 w[4];
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[q] = bm4[tid * 4 + q];
      cnt += __popc(w[q].x) + __popc(w[q].y) + __popc(w[q].z) + __popc(w[q].w);
    }
    uint32_t pos = written + block_excl_sum(cnt, scan_buf);
    const uint32_t total = scan_buf[kMergeWarps - 1];
    if (cnt) {
      const uint32_t id0 = c0 + static_cast<uint32_t>(tid) * 512u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t m = ws[e];
          while (m) {
            const int b = __ffs(m) - 1;
            m &= m - 1;
            if (pos < static_cast<uint32_t>(k)) orow[pos] = static_cast<int32_t>(id0 + (q * 4 + e) * 32 + b);
            ++pos;
          }
        }
      }
    }
    written += total;
    __syncthreads();
  }
  for (int i = static_cast<int>(min(written, static_cast<uint32_t>(k))) + tid; i < k; i += kMergeThreads) orow[i] = -1;
}

}  // namespace

cudaError_t launch_dcp_pack(const void* logits, int32_t logits_dtype, int64_t logits_stride,
                            const int32_t* local_idx, int64_t idx_stride, int32_t num_rows, int32_t k,
                            int32_t rank, int32_t world, int32_t interleave, float* packed,
                            cudaStream_t stream) {
  float2* po = reinterpret_cast<float2*>(packed);
  if (logits_dtype == DSA_LOGITS_BF16)
    pack_kernel<__nv_bfloat16><<<num_rows, kPackThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(logits),
                                                             logits_stride, local_idx, idx_stride, k,
                                                             rank, world, interleave, po);
  else
    pack_kernel<float><<<num_rows, kPackThreads, 0, stream>>>(static_cast<const float*>(logits), logits_stride,
                                                     local_idx, idx_stride, k, rank, world, interleave, po);
  return cudaGetLastError();
}

cudaError_t launch_dcp_merge(const float* gathered, int32_t world, int32_t num_rows, int32_t k,
                             int32_t* out_idx, int64_t out_stride, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
  if (e != cudaSuccess) return e;
  merge_kernel<<<num_rows, kMergeThreads, kMergeSmem, stream>>>(reinterpret_cast<const float2*>(gathered), world,
                                                                num_rows, k, out_idx, out_stride);
  return cudaGetLastError();
}

}  // namespace dsa
