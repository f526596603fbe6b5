// Work schedule of the logits kernel (the metadata call of PR 47469 "Route
// SM100 sparse-indexer decode through varlen paged MQA logits", Purpose and
// Changes: get_paged_mqa_logits_metadata(seq_lens, block_kv, num_sms,
// indices) -> SM schedule; rows with equal consecutive request ids belong to
// one request, PR 56811 "Fix fp8_fp4_paged_mqa_logits MQA kpool varlen path
// for speculative decode", Purpose).  The pages fix the call's inputs and its
// purpose, balancing (request, K-block) work over the SMs; the split rule is
// this library's own.
//
// A unit is one 128-key tile of one group (up to 8 adjacent rows of one
// request).  It costs its SM one K tile from HBM, the same for every unit,
// plus MMA columns and epilogue work that grow with the group's rows: a unit
// of n rows weighs unit_weight(format, n) (n for FP4 keys, 4n + n^2 for FP8
// and MXFP4, whose tiles cost more than linearly in their rows).  The
// rule gives every SM the same number of units (within one) and, as nearly
// as the groups allow, the same weight:
//   1. groups: runs of equal request ids, each cut into pieces of at most
//      group_rows_for(format) rows;
//   2. the groups are ordered by row count (stable) and their units laid end
//      to end in that order: sorted position k starts at unit sus[k], and
//      spp[k] weight precedes it;
//   3. boundary i (0 <= i <= S) has consumed x_i = floor(i U / S) units,
//      lambda_i from the light (left) end of that sequence and
//      x_i - lambda_i from the heavy (right) end; SM i owns the units between
//      boundaries i and i + 1 at both ends;
//   4. a_i = the fewest left units such that the weight consumed, times S,
//      does not exceed i P (P = all weight), and lambda_i is a_i moved as
//      little as needed to keep both ends monotone: lambda_i =
//      max(lambda_{i-1}, min(a_i, lambda_{i-1} + x_i - x_{i-1})).
//
// One CTA (256 threads; 1024 for 256 SMs or more, or more than 1024 rows):
// chunked block scans for the groups, the stable counting sort by row count
// and the prefix sums; one thread per boundary for a_i; thread 0 for the
// monotone pass.  The groups of one row count n are adjacent in the sorted
// order and their units weigh the same, so the weight before unit u is
// piecewise linear in u with one piece per row count, and so is the weight
// consumed at boundary i as a function of the left units: a_i is solved
// exactly from its values where either end enters a new piece
// (ClassPieces::fewest_left).  ("pairs" in the code below is that weight.)
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

// Block sizes: 256 threads (8 warps: shorter barriers and scans) when there
// are fewer than 256 SMs to split over and at most 1024 rows, else 1024; a
// boundary takes one thread.
constexpr int kThreadsSmall = 256;
constexpr int kThreadsLarge = 1024;

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

// Exclusive prefix sum over a block of kW warps; *total receives the block sum.
template <int kW, typename T>
__device__ T block_exclusive_sum(T v, T* buf, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T inc = warp_inclusive_sum(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T s = lane < kW ? buf[lane] : T(0);
    s = warp_inclusive_sum(s);
    if (lane < kW) buf[lane] = s;
  }
  __syncthreads();
  const T before = warp ? buf[warp - 1] : T(0);
  *total = buf[kW - 1];
  __syncthreads();
  return before + inc - v;
}

// Two exclusive prefix sums over the block with the barriers of one.
template <int kW, typename A, typename B>
__device__ void block_exclusive_sum2(A va, B vb, A* bufa, B* bufb, A& exa, B& exb, A& tota, B& totb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const A ia = warp_inclusive_sum(va);
  const B ib = warp_inclusive_sum(vb);
  if (lane == 31) {
    bufa[warp] = ia;
    bufb[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const A sa = warp_inclusive_sum(lane < kW ? bufa[lane] : A(0));
    const B sb = warp_inclusive_sum(lane < kW ? bufb[lane] : B(0));
    if (lane < kW) {
      bufa[lane] = sa;
      bufb[lane] = sb;
    }
  }
  __syncthreads();
  exa = (warp ? bufa[warp - 1] : A(0)) + ia - va;
  exb = (warp ? bufb[warp - 1] : B(0)) + ib - vb;
  tota = bufa[kW - 1];
  totb = bufb[kW - 1];
  __syncthreads();
}

template <int kW>
__device__ int block_inclusive_max(int v, int* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int inc = warp_inclusive_max(v);
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int m = warp_inclusive_max(lane < kW ? buf[lane] : INT_MIN);
    if (lane < kW) buf[lane] = m;
  }
  __syncthreads();
  const int r = warp ? max(inc, buf[warp - 1]) : inc;
  __syncthreads();
  return r;
}

// Rows up to which the working arrays (group starts, sorted positions, unit
// starts, pair prefixes) live in dynamic shared memory; the kernel copies them
// to the schedule at the end.  Larger batches work on the schedule words in
// global memory directly (the block's own global writes are visible to it
// after __syncthreads).
constexpr int kSmemRows = 8192;
constexpr int kSchedArrays = 5;  // grs, pos, sus, spp_lo, spp_hi

// The sorted unit sequence as one linear piece per row count n = 1 ..
// kGroupMaxRows: units [u0[n], u0[n + 1]) weigh wt[n] each, p0[n] before the
// first of them (u0 non-decreasing, u0[1] = 0; an empty piece
// starts where the next one does).
struct ClassPieces {
  int32_t u0[kGroupMaxRows + 1];  // in registers: the thresholds
  const int32_t* su0;             // shared copies, indexed by row count
  const int64_t* sp0;
  const int64_t* swt;             // weight of one unit of each piece

  // Pairs of the first u units (0 <= u <= U): the piece holding unit u is the
  // last one starting at or before u, i.e. the number of pieces that do.
  __device__ __forceinline__ int64_t pairs_before(int32_t u) const {
    int n = 0;
#pragma unroll
    for (int c = 1; c <= kGroupMaxRows; ++c) n += u >= u0[c] ? 1 : 0;
    return sp0[n] + static_cast<int64_t>(u - su0[n]) * swt[n];
  }

  // The fewest left units lam in [0, x] with pairs consumed <= cap, x if
  // none.  The pairs consumed, f(lam) = pairs_before(lam) + P -
  // pairs_before(U - x + lam), do not increase with lam and are linear
  // between the points where either end enters a new piece: lam = u0[c]
  // (there pairs_before(lam) = p0[c]) and lam = u0[c] - (U - x) (there the
  // right term is p0[c]).  f at those points (independent evaluations) gives
  // the last point above cap and the first at or below it; between the two f
  // falls by a whole number of pairs per unit, which gives lam exactly.
  __device__ __forceinline__ int32_t fewest_left(int32_t x, int32_t U, int64_t P, int64_t cap) const {
    const int32_t off = U - x;  // the right end is off + lam
    const int64_t f0 = P - pairs_before(off);
    if (f0 <= cap) return 0;
    const int64_t fx = pairs_before(x);  // + P - pairs_before(U)
    if (fx > cap) return x;
    int32_t blo = 0, bhi = x;  // last point above cap, first at or below
    int64_t flo = f0, fhi = fx;
#pragma unroll
    for (int c = 2; c <= kGroupMaxRows; ++c) {
      const int32_t bl = u0[c], br = u0[c] - off;
      const bool inl = bl > 0 && bl < x, inr = br > 0 && br < x;
      const int64_t fl = sp0[c] + P - pairs_before(inl ? off + bl : 0);
      const int64_t fr = pairs_before(inr ? br : 0) + P - sp0[c];
      if (inl) {
        if (fl > cap) {
          if (bl > blo) { blo = bl; flo = fl; }
        } else if (bl < bhi) {
          bhi = bl;
          fhi = fl;
        }
      }
      if (inr) {
        if (fr > cap) {
          if (br > blo) { blo = br; flo = fr; }
        } else if (br < bhi) {
          bhi = br;
          fhi = fr;
        }
      }
    }
    // f falls by d = (unit weight at the right end) - (unit weight at the
    // left end) a unit, d >= 1; both divisions in 32 bits when the operands
    // fit (a 64-bit division costs ~1.5K cycles)
    const uint64_t num = static_cast<uint64_t>(flo - fhi), den = static_cast<uint64_t>(bhi - blo);
    const uint32_t d = (num >> 32) == 0 ? static_cast<uint32_t>(num) / static_cast<uint32_t>(den)
                                        : static_cast<uint32_t>(num / den);
    const uint64_t q = static_cast<uint64_t>(flo - cap) + d - 1;
    const uint64_t steps = (q >> 32) == 0 ? static_cast<uint32_t>(q) / d : q / d;
    return blo + static_cast<int32_t>(steps);
  }
};

// kInSmem: the working arrays live in dynamic shared memory (T <= kSmemRows)
// and every pointer to them is derived from that array, so that their loads
// and stores are shared-memory accesses; otherwise they are the schedule's
// own words in global memory.
template <bool kInSmem, int kThreads>
__global__ void __launch_bounds__(kThreads, 1)
    metadata_kernel(const int32_t* __restrict__ ctx, const int32_t* __restrict__ ind, int32_t T,
                    int32_t S, int32_t kv_format, int32_t* __restrict__ sched) {
  // the logits kernel launched after this one may start its set-up now
  grid_dep_launch();
  constexpr int kWarps = kThreads / 32;
  extern __shared__ int32_t dyn[];
  __shared__ int32_t buf32[kWarps];
  __shared__ int64_t buf64[kWarps];
  __shared__ uint64_t bufu[kWarps];
  __shared__ uint64_t bufu2[kWarps];
  __shared__ int32_t s_carry;
  __shared__ int32_t s_base[kGroupMaxRows + 1];   // first sorted position of each row count
  __shared__ int32_t s_taken[kGroupMaxRows + 1];  // positions of each row count handed out so far
  __shared__ int32_t s_a[kThreads];
  __shared__ int32_t s_x[kThreads];
  __shared__ int32_t s_lambda[kThreads];
  __shared__ int32_t s_u0[kGroupMaxRows + 1];  // first unit of each row count's piece
  __shared__ int64_t s_p0[kGroupMaxRows + 1];  // weight before it
  __shared__ int64_t s_wt[kGroupMaxRows + 1];  // weight of one unit of the piece
  __shared__ int64_t s_pq, s_pr;                // P = s_pq * S + s_pr
  __shared__ int32_t s_ctx[kThreads];           // causal limits when T <= kThreads

  const int tid = threadIdx.x;
  const SchedLayout L(S, T);
  const int group_rows = group_rows_for(kv_format);
  const int64_t n1 = static_cast<int64_t>(T) + 1;
  int32_t* const base = kInSmem ? dyn : sched + L.grs;  // the five arrays, end to end, in both places
  int32_t* grs = base;
  int32_t* pos = base + n1;
  int32_t* sus = base + 2 * n1;
  int32_t* spp_lo = base + 3 * n1;
  int32_t* spp_hi = base + 4 * n1;
  // ---- groups: a row starts one when it starts a run of equal request ids,
  // or when group_rows (<= kGroupMaxRows) rows of its run precede it in the current group
  // When the rows fit one pass of the block, each thread's causal limit is
  // loaded now (in flight during the groups phase) and kept in shared memory
  // for the units phase, which would otherwise wait on a second global load.
  const bool one_chunk = T <= kThreads;
  const int32_t my_ctx = (one_chunk && tid < T) ? __ldg(ctx + tid) : 0;
  int carry_run = 0;  // run start of the previous chunk's last row
  int G = 0;
  for (int base = 0; base < T; base += kThreads) {
    const int t = base + tid;
    const bool valid = t < T;
    const bool run_start = valid && (t == 0 || ind == nullptr || ind[t] != ind[t - 1]);
    int rs = block_inclusive_max<kWarps>(run_start ? t : -1, buf32);
    rs = max(rs, carry_run);
    const bool gstart = valid && ((t - rs) % group_rows == 0);
    int32_t total;
    const int32_t idx = block_exclusive_sum<kWarps, int32_t>(gstart ? 1 : 0, buf32, &total);
    if (gstart) grs[G + idx] = t;
    G += total;
    if (tid == kThreads - 1) s_carry = rs;
    __syncthreads();
    carry_run = s_carry;
    __syncthreads();
  }
  for (int g = G + tid; g <= T; g += kThreads) grs[g] = T;
  if (one_chunk) s_ctx[tid] = my_ctx;
  if (tid <= kGroupMaxRows) {
    s_base[tid] = 0;
    s_taken[tid] = 0;
  }
  __syncthreads();

  // ---- stable counting sort of the groups by row count (1 .. kGroupMaxRows)
  for (int g = tid; g < G; g += kThreads) atomicAdd(&s_base[grs[g + 1] - grs[g]], 1);
  __syncthreads();
  if (tid == 0) {
    int b = 0;
    for (int n = 1; n <= kGroupMaxRows; ++n) {
      const int c = s_base[n];
      s_base[n] = b;
      b += c;
    }
  }
  __syncthreads();
  // ranks within a row count: one-hot counters, 16 bits each, four counts per
  // 64-bit scan (a chunk holds at most 1024 groups)
  static_assert(kGroupMaxRows == 8 && kThreads < 65536, "packed rank counters");
  for (int base = 0; base < G; base += kThreads) {
    const int g = base + tid;
    const bool valid = g < G;
    const int n = valid ? grs[g + 1] - grs[g] : 0;
    const uint64_t one_lo = (valid && n <= 4) ? (1ull << (16 * (n - 1))) : 0ull;
    const uint64_t one_hi = (valid && n > 4) ? (1ull << (16 * (n - 5))) : 0ull;
    uint64_t tot_lo, tot_hi, ex_lo, ex_hi;
    block_exclusive_sum2<kWarps, uint64_t, uint64_t>(one_lo, one_hi, bufu, bufu2, ex_lo, ex_hi, tot_lo, tot_hi);
    if (valid) {
      const int rank = static_cast<int>(n <= 4 ? (ex_lo >> (16 * (n - 1))) & 0xffffu : (ex_hi >> (16 * (n - 5))) & 0xffffu);
      pos[s_base[n] + s_taken[n] + rank] = grs[g] | (n << kPosRowsShift);
    }
    __syncthreads();
    if (tid < kGroupMaxRows) {
      const int cls = tid + 1;
      s_taken[cls] += static_cast<int>(cls <= 4 ? (tot_lo >> (16 * (cls - 1))) & 0xffffu : (tot_hi >> (16 * (cls - 5))) & 0xffffu);
    }
    __syncthreads();
  }

  // ---- units and pairs along the sorted order
  int32_t U = 0;
  int64_t P = 0;
  for (int base = 0; base < G; base += kThreads) {
    const int k = base + tid;
    int32_t tiles = 0;
    int64_t pairs = 0;
    if (k < G) {
      const int32_t w = pos[k];
      const int r0 = w & kPosRowMask, n = static_cast<int>(static_cast<uint32_t>(w) >> kPosRowsShift);
      // the group's largest causal limit: all its loads in flight at once
      int lmax = 0;
#pragma unroll
      for (int j = 0; j < kGroupMaxRows; ++j)
        if (j < n) lmax = max(lmax, one_chunk ? s_ctx[r0 + j] : __ldg(ctx + r0 + j));
      tiles = (lmax + kTileTokens - 1) / kTileTokens;
      pairs = static_cast<int64_t>(tiles) * unit_weight(kv_format, n);
    }
    int32_t tot, ex;
    int64_t totp, exp;
    block_exclusive_sum2<kWarps, int32_t, int64_t>(tiles, pairs, buf32, buf64, ex, exp, tot, totp);
    if (k < G) {
      sus[k] = U + ex;
      const int64_t pp = P + exp;
      spp_lo[k] = static_cast<int32_t>(pp & 0xffffffff);
      spp_hi[k] = static_cast<int32_t>(pp >> 32);
    }
    U += tot;
    P += totp;
  }

  for (int k = G + tid; k <= T; k += kThreads) {
    pos[k] = T;  // past the last group
    sus[k] = U;
    spp_lo[k] = static_cast<int32_t>(P & 0xffffffff);
    spp_hi[k] = static_cast<int32_t>(P >> 32);
  }
  __syncthreads();

  // ---- the pieces: row count n starts at sorted position s_base[n]
  if (tid >= 1 && tid <= kGroupMaxRows) {
    s_wt[tid] = unit_weight(kv_format, tid);
    const int k = s_base[tid];
    s_u0[tid] = sus[k];
    s_p0[tid] = static_cast<int64_t>(static_cast<uint32_t>(spp_lo[k])) | (static_cast<int64_t>(spp_hi[k]) << 32);
  }
  if (tid == 0) {
    s_u0[0] = 0;
    s_p0[0] = 0;
    s_wt[0] = 0;
    // (a 64-bit division costs ~1.5K cycles: 32 bits when P fits)
    if ((static_cast<uint64_t>(P) >> 32) == 0) {
      const uint32_t p32 = static_cast<uint32_t>(P), s32 = static_cast<uint32_t>(S);
      s_pq = p32 / s32;
      s_pr = p32 - (p32 / s32) * s32;
    } else {
      s_pq = P / S;
      s_pr = P % S;
    }
  }
  __syncthreads();

  // ---- a_i: the fewest left units with (pairs consumed) * S <= i * P
  if (tid <= S) {
    // x = floor(i U / S) and cap = floor(i P / S) without a wide division:
    // U = q S + r gives i U / S = i q + (i r) / S with i r < 2^20
    const int32_t uq = U / S, ur = U - uq * S;
    const int32_t x = tid * uq + (tid * ur) / S;
    s_x[tid] = x;
    // i (P mod S) < S^2 < 2^20: a 32-bit division
    const int64_t cap = static_cast<int64_t>(tid) * s_pq +
                        static_cast<int64_t>(static_cast<uint32_t>(tid * static_cast<int32_t>(s_pr)) /
                                             static_cast<uint32_t>(S));
    ClassPieces cp;
#pragma unroll
    for (int n = 1; n <= kGroupMaxRows; ++n) cp.u0[n] = s_u0[n];
    cp.su0 = s_u0;
    cp.sp0 = s_p0;
    cp.swt = s_wt;
    s_a[tid] = cp.fewest_left(x, U, P, cap);
  }
  __syncthreads();

  // ---- monotone path: lambda_i = max(lambda_{i-1}, min(a_i, lambda_{i-1} +
  // x_i - x_{i-1})).  Where no step of the running maximum of a exceeds its
  // x step, that running maximum is the path (one block-wide max scan);
  // otherwise thread 0 walks the recurrence.
  {
    const int a = tid <= S ? s_a[tid] : 0;
    const int run = block_inclusive_max<kWarps>(a, buf32);
    if (tid <= S) s_lambda[tid] = run;
    __syncthreads();
    const bool bad = tid >= 1 && tid <= S && s_lambda[tid] - s_lambda[tid - 1] > s_x[tid] - s_x[tid - 1];
    const int any_bad = __syncthreads_or(bad ? 1 : 0);
    if (any_bad && tid == 0) {
      int32_t lam = 0;
      s_lambda[0] = 0;
      for (int i = 1; i <= S; ++i) {
        lam = max(lam, min(s_a[i], lam + (s_x[i] - s_x[i - 1])));
        s_lambda[i] = lam;
      }
    }
    __syncthreads();
  }
  if (tid <= S) {
    sched[L.left + tid] = s_lambda[tid];
    sched[L.right + tid] = U - (s_x[tid] - s_lambda[tid]);
  }
  if (kInSmem) {  // the working arrays to the schedule
    for (int64_t i = tid; i < kSchedArrays * n1; i += kThreads) sched[L.grs + i] = dyn[i];
  }
  if (tid == 0) {
    sched[0] = kScheduleMagic;
    sched[1] = T;
    sched[2] = ind != nullptr ? 1 : 0;
    sched[3] = S;
    sched[4] = G;
    sched[5] = U;
    sched[6] = kTileTokens;
    sched[7] = group_rows;
  }
}

}  // namespace

namespace {

template <int kThreads>
cudaError_t launch_metadata_as(const int32_t* context_lens, const int32_t* indices, int32_t num_rows,
                               int32_t num_sms, int32_t kv_format, int32_t* schedule, cudaStream_t stream) {
  if (num_rows > kSmemRows) {
    metadata_kernel<false, kThreads><<<1, kThreads, 0, stream>>>(context_lens, indices, num_rows, num_sms,
                                                                  kv_format, schedule);
    return cudaGetLastError();
  }
  const size_t smem = kSchedArrays * (static_cast<size_t>(num_rows) + 1) * 4;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(metadata_kernel<true, kThreads>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSchedArrays * (kSmemRows + 1) * 4);
    if (e != cudaSuccess) return e;
  }
  metadata_kernel<true, kThreads><<<1, kThreads, smem, stream>>>(context_lens, indices, num_rows, num_sms,
                                                                 kv_format, schedule);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_metadata(const int32_t* context_lens, const int32_t* indices, int32_t num_rows,
                            int32_t num_sms, int32_t kv_format, int32_t* schedule, cudaStream_t stream) {
  static_assert(kSchedArrays * (kSmemRows + 1) * 4 <= 200 * 1024, "metadata shared memory");
  // one thread per boundary 0 .. num_sms; many rows (prefill chunks) take the
  // large block, whose scans cover 1024 rows a pass
  if (num_sms < kThreadsSmall && num_rows <= kThreadsLarge)
    return launch_metadata_as<kThreadsSmall>(context_lens, indices, num_rows, num_sms, kv_format, schedule, stream);
  return launch_metadata_as<kThreadsLarge>(context_lens, indices, num_rows, num_sms, kv_format, schedule, stream);
}

}  // namespace dsa
