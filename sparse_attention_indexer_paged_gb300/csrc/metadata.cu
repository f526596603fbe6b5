// Work schedule of the logits kernel (the metadata call of PR 47469 "Route
// SM100 sparse-indexer decode through varlen paged MQA logits", Purpose and
// Changes: get_paged_mqa_logits_metadata(seq_lens, block_kv, num_sms,
// indices) -> SM schedule; rows with equal consecutive request ids belong to
// one request, PR 56811 "Fix fp8_fp4_paged_mqa_logits MQA kpool varlen path
// for speculative decode", Purpose).
//
// One CTA of 1024 threads walks the rows and groups in chunks of 1024 with
// block-wide scans:
//   pass 1  group starts: a row starts a group when it starts a run of equal
//           request ids, or when kGroupMaxRows rows of its run precede it in
//           the current group;
//   pass 2  tiles per group = ceil(max L_t / 128) and their prefix sums;
//   pass 3  prefix weights (tile weight = kTileWeight + kRowWeight * rows) and, for every
//           SM i, the first tile u with P(u) * num_sms >= i * W (exact
//           integer arithmetic).
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

template <typename T>
__device__ __forceinline__ T warp_inclusive_sum(T x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ int warp_inclusive_max(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  return x;
}

// Exclusive prefix sum over the block; *total receives the block sum.
template <typename T>
__device__ T block_exclusive_sum(T v, T* buf, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T inc = warp_inclusive_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T s = buf[lane];
    s = warp_inclusive_sum(s);
    buf[lane] = s;
  }
  __syncthreads();
  const T before = warp ? buf[warp - 1] : T(0);
  *total = buf[kWarps - 1];
  __syncthreads();
  return before + inc - v;
}

__device__ int block_inclusive_max(int v, int* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int inc = warp_inclusive_max(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) buf[lane] = warp_inclusive_max(buf[lane]);
  __syncthreads();
  const int r = warp ? max(inc, buf[warp - 1]) : inc;
  __syncthreads();
  return r;
}

struct GroupInfo {
  int32_t tiles;
  int32_t weight;
};

__device__ __forceinline__ GroupInfo group_info(const int32_t* ctx, const int32_t* grs, int g,
                                                int G, int T) {
  const int r0 = grs[g];
  const int r1 = (g + 1 < G) ? grs[g + 1] : T;
  int lmax = 0;
  for (int t = r0; t < r1; ++t) lmax = max(lmax, ctx[t]);
  GroupInfo gi;
  gi.tiles = (lmax + kTileTokens - 1) / kTileTokens;
  gi.weight = kTileWeight + kRowWeight * (r1 - r0);
  return gi;
}

__global__ void __launch_bounds__(kThreads, 1)
    metadata_kernel(const int32_t* __restrict__ ctx, const int32_t* __restrict__ ind, int32_t T,
                    int32_t S, int32_t* __restrict__ sched) {
  __shared__ int32_t buf32[kWarps];
  __shared__ int64_t buf64[kWarps];
  __shared__ int64_t s_key[kThreads];
  __shared__ int64_t s_gw[kThreads];
  __shared__ int32_t s_us[kThreads];
  __shared__ int32_t s_w[kThreads];
  __shared__ int32_t s_carry;

  const int tid = threadIdx.x;
  int32_t* sm_start = sched + kScheduleHeaderWords;
  int32_t* grs = sm_start + S + 1;
  int32_t* gus = grs + T + 1;

  // ---- pass 1: group starts
  int carry_run = 0;  // run start of the previous chunk's last row
  int G = 0;
  for (int base = 0; base < T; base += kThreads) {
    const int t = base + tid;
    const bool valid = t < T;
    const bool run_start = valid && (t == 0 || ind == nullptr || ind[t] != ind[t - 1]);
    int rs = block_inclusive_max(run_start ? t : -1, buf32);
    rs = max(rs, carry_run);
    const bool gstart = valid && ((t - rs) % kGroupMaxRows == 0);
    int32_t total;
    const int32_t idx = block_exclusive_sum<int32_t>(gstart ? 1 : 0, buf32, &total);
    if (gstart) grs[G + idx] = t;
    G += total;
    if (tid == kThreads - 1) s_carry = rs;
    __syncthreads();
    carry_run = s_carry;
    __syncthreads();
  }
  for (int g = G + tid; g <= T; g += kThreads) grs[g] = T;
  __syncthreads();

  // ---- pass 2: tiles per group and their prefix sums
  int U = 0;
  int64_t W = 0;
  for (int base = 0; base < G; base += kThreads) {
    const int g = base + tid;
    GroupInfo gi{0, 0};
    if (g < G) gi = group_info(ctx, grs, g, G, T);
    int32_t tot;
    const int32_t ex = block_exclusive_sum<int32_t>(gi.tiles, buf32, &tot);
    int64_t totw;
    block_exclusive_sum<int64_t>(static_cast<int64_t>(gi.tiles) * gi.weight, buf64, &totw);
    if (g < G) gus[g] = U + ex;
    U += tot;
    W += totw;
  }
  for (int g = G + tid; g <= T; g += kThreads) gus[g] = U;
  __syncthreads();

  // ---- pass 3: SM boundaries.  Thread i owns boundary i (i <= S).
  const int64_t target = static_cast<int64_t>(tid) * W;  // compare P(u) * S >= target
  bool resolved = tid > S;
  int32_t answer = U;
  int unit_carry = 0;
  int64_t weight_carry = 0;
  for (int base = 0; base < G; base += kThreads) {
    const int g = base + tid;
    GroupInfo gi{0, 0};
    if (g < G) gi = group_info(ctx, grs, g, G, T);
    int32_t tot;
    const int32_t ex = block_exclusive_sum<int32_t>(gi.tiles, buf32, &tot);
    int64_t totw;
    const int64_t exw =
        block_exclusive_sum<int64_t>(static_cast<int64_t>(gi.tiles) * gi.weight, buf64, &totw);
    const int64_t gw = weight_carry + exw;
    // key = weight before the group's last tile (empty group: gw - 1), so keys
    // never decrease along the groups; padding entries are +inf.
    s_key[tid] = (g < G) ? (gi.tiles > 0 ? gw + static_cast<int64_t>(gi.tiles - 1) * gi.weight
                                         : gw - 1)
                         : INT64_MAX;
    s_gw[tid] = gw;
    s_us[tid] = unit_carry + ex;
    s_w[tid] = gi.weight;
    __syncthreads();
    const int n_in = min(kThreads, G - base);
    if (!resolved && s_key[n_in - 1] * S >= target) {
      int lo = 0, hi = n_in - 1;  // first index with key * S >= target
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_key[mid] * S >= target) hi = mid; else lo = mid + 1;
      }
      const int64_t num = target - s_gw[lo] * S;
      const int64_t den = static_cast<int64_t>(s_w[lo]) * S;
      const int64_t add = num > 0 ? (num + den - 1) / den : 0;
      answer = s_us[lo] + static_cast<int32_t>(add);
      resolved = true;
    }
    __syncthreads();
    unit_carry += tot;
    weight_carry += totw;
  }
  if (tid <= S) sm_start[tid] = (W == 0) ? 0 : answer;
  if (tid == 0) {
    sched[0] = kScheduleMagic;
    sched[1] = T;
    sched[2] = ind != nullptr ? 1 : 0;
    sched[3] = S;
    sched[4] = G;
    sched[5] = U;
    sched[6] = kTileTokens;
    sched[7] = kGroupMaxRows;
  }
}

}  // namespace

cudaError_t launch_metadata(const int32_t* context_lens, const int32_t* indices, int32_t num_rows,
                            int32_t num_sms, int32_t* schedule, cudaStream_t stream) {
  metadata_kernel<<<1, kThreads, 0, stream>>>(context_lens, indices, num_rows, num_sms, schedule);
  return cudaGetLastError();
}

}  // namespace dsa
