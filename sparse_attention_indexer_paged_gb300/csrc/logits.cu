// Varlen paged MQA logits for sm_103a (PR 47469 "Route SM100 sparse-indexer
// decode through varlen paged MQA logits", Purpose; PR 56811 "Fix
// fp8_fp4_paged_mqa_logits MQA kpool varlen path for speculative decode",
// Purpose; sparse_attn_indexer docs, _varlen_decode_rows):
//
//   logits[t, s] = kscale[s] * sum_h w[t, h] * relu(sum_d q[t, h, d] * k[s, d])
//
// One persistent CTA per SM walks the (group, tile) units the metadata call
// gave it.  A group is up to 8 adjacent rows of one request; a tile is 128
// keys (two 64-token pages).  Every K tile is read from HBM once per group
// and serves all of the group's rows and heads.
//
// The contraction is laid out with the keys as M: for each tile and each
// row r of the group, D[token, h] = sum_d K[token, d] * Q[r, h, d] is one
// 128 x 64 block of a tcgen05 MMA (A = the K tile, B = the group's Q rows,
// N = 64 per row, up to 4 rows per instruction).  TMEM lane = token, so the
// head-weighted ReLU reduction of a (token, row) runs inside one thread with
// no cross-lane traffic, and a warp's 32 logits are 32 consecutive columns.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: the group's Q rows and weights, then the K
//               pages (3-D tensor map over the pool, page id from the block
//               table) and their scales, into a kStages-deep ring.
//   warp 1      MMA issuer and TMEM owner (512 columns = 8 slots of 64).
//   warps 2-3   idle (FP8) / key dequantisation (FP4).
//   warps 4-11  two epilogue warpgroups: tcgen05.ld of a (tile, row) slot,
//               relu, packed-fp32 FMA with the head weights, key scale,
//               causal mask, store.  Warpgroup g drains the TMEM slots of
//               parity g, so every slot barrier has a single consumer that
//               sees each of its phases in order (a parity wait cannot then
//               pass on a phase that belongs to another consumer).
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 384;
constexpr int kStages = 6;
constexpr int kTmemCols = 512;
constexpr int kSlots = 8;
constexpr int kSlotCols = 64;
constexpr int kMaxRowsPerMma = 4;  // N = 256

constexpr int kPageValBytesFp8 = kPageTokens * kHeadDim;  // 8192
constexpr int kKvStageBytes = 2 * kPageValBytesFp8;       // 16384: one 128 x 128 e4m3 tile
constexpr int kQRowBytes = kHeads * kHeadDim;             // 8192: 64 heads x 128 e4m3
constexpr int kScaleStageFloats = kTileTokens;            // 128 key scales per tile
constexpr int kWBufFloats = kGroupMaxRows * kHeads;       // 512

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffKv = 0;
constexpr int kOffQ = kOffKv + kStages * kKvStageBytes;
constexpr int kOffScale = kOffQ + kGroupMaxRows * kQRowBytes;
constexpr int kOffW = kOffScale + kStages * kScaleStageFloats * 4;
constexpr int kOffBar = kOffW + 2 * kWBufFloats * 4;
// barriers: kv_full[S], kv_empty[S], q_full, q_empty, w_full[2], w_empty[2],
// tmem_full[8], tmem_empty[8], mma_done
constexpr int kNumBars = 2 * kStages + 2 + 4 + 2 * kSlots + 1;
constexpr int kOffTmemAddr = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemAddr + 4;
constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kOffQ % 1024 == 0 && kOffKv % 1024 == 0, "MMA tiles need 1024-byte alignment");
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");

struct Params {
  const uint8_t* kv_cache;
  int64_t page_stride;
  int64_t num_pages;
  const float* weights;
  const int32_t* ctx;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* indices;
  const int32_t* schedule;
  int32_t num_sms;
  void* logits;
  int32_t logits_bf16;
  int64_t logits_stride;
  int32_t num_rows;
  int32_t* status;
};

struct Bars {
  uint32_t kv_full, kv_empty, q_full, q_empty, w_full, w_empty, tmem_full, tmem_empty, mma_done;
  __device__ uint32_t kvf(int s) const { return kv_full + 8 * s; }
  __device__ uint32_t kve(int s) const { return kv_empty + 8 * s; }
  __device__ uint32_t wf(int b) const { return w_full + 8 * b; }
  __device__ uint32_t we(int b) const { return w_empty + 8 * b; }
  __device__ uint32_t tf(int s) const { return tmem_full + 8 * s; }
  __device__ uint32_t te(int s) const { return tmem_empty + 8 * s; }
};

// The CTA's walk over its units: groups in order, and the tiles [j0, j1) of
// each group that belong to this CTA.  Every role runs the same walk.
struct Walk {
  const int32_t* grs;
  const int32_t* gus;
  const int32_t* ctx;
  int G, T, u, u_end, g;
  // current group
  int r0, n, npages, j0, j1;

  __device__ void start(const int32_t* grs_, const int32_t* gus_, const int32_t* ctx_, int G_,
                        int T_, int u0, int u1) {
    T = T_;
    grs = grs_;
    gus = gus_;
    ctx = ctx_;
    G = G_;
    u = u0;
    u_end = u1;
    // largest g with gus[g] <= u
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (gus[mid] <= u) lo = mid; else hi = mid - 1;
    }
    g = lo;
  }

  // Loads the next group that holds units of this CTA; false when done.
  __device__ bool next() {
    while (u < u_end && g < G && gus[g + 1] <= u) ++g;
    if (u >= u_end || g >= G) return false;
    const int gu0 = gus[g];
    r0 = grs[g];
    n = grs[g + 1] - r0;
    if (r0 < 0 || n <= 0 || n > kGroupMaxRows || r0 + n > T) return false;
    int lmax = 0;
    for (int t = r0; t < r0 + n; ++t) lmax = max(lmax, ctx[t]);
    npages = (lmax + kPageTokens - 1) / kPageTokens;
    j0 = u - gu0;
    j1 = min(gus[g + 1], u_end) - gu0;
    u = gu0 + j1;
    return true;
  }
};

// Warp-uniform wait: lane 0 waits (bounded), the verdict is broadcast, and
// every lane then observes the completed phase itself (it cannot move on
// before this warp arrives on the matching "empty" barrier).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) {
    for (int i = 0; i < (1 << 20) && !mbar_try_wait(bar, parity); ++i) {
    }
  }
  return ok != 0;
}

__device__ __forceinline__ float relu_f(uint32_t bits) { return fmaxf(__uint_as_float(bits), 0.0f); }

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                  const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- the schedule must be the one built for these rows, mode and SM count
  const int32_t* sched = p.schedule;
  const int S = p.num_sms;
  const int T = p.num_rows;
  if (sched[0] != kScheduleMagic || sched[1] != T || sched[2] != (p.indices != nullptr ? 1 : 0) ||
      sched[3] != S || sched[6] != kTileTokens || sched[7] != kGroupMaxRows ||
      static_cast<int>(gridDim.x) != S || sched[4] < 0 || sched[4] > T) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(p.status, kErrScheduleMismatch);
    return;
  }
  const int G = sched[4];
  const int U = sched[5];
  const int32_t* sm_start = sched + kScheduleHeaderWords;
  const int32_t* grs = sm_start + S + 1;
  const int32_t* gus = grs + T + 1;
  const int u0 = min(max(sm_start[blockIdx.x], 0), U);
  const int u1 = min(max(sm_start[blockIdx.x + 1], u0), U);
  if (u0 >= u1 || G == 0) return;  // no work: the whole CTA leaves before any set-up

  Bars bars;
  const uint32_t bar0 = sbase + kOffBar;
  bars.kv_full = bar0;
  bars.kv_empty = bars.kv_full + 8 * kStages;
  bars.q_full = bars.kv_empty + 8 * kStages;
  bars.q_empty = bars.q_full + 8;
  bars.w_full = bars.q_empty + 8;
  bars.w_empty = bars.w_full + 16;
  bars.tmem_full = bars.w_empty + 16;
  bars.tmem_empty = bars.tmem_full + 8 * kSlots;
  bars.mma_done = bars.tmem_empty + 8 * kSlots;
  uint32_t* tmem_addr_smem = reinterpret_cast<uint32_t*>(smem + kOffTmemAddr);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars.kvf(s), 1);
      mbar_init(bars.kve(s), 1 + 8);  // MMA commit + every epilogue warp (key scales read)
    }
    mbar_init(bars.q_full, 1);
    mbar_init(bars.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.wf(b), 1);
      mbar_init(bars.we(b), 8);  // every epilogue warp
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bars.tf(s), 1);
      mbar_init(bars.te(s), 4);
    }
    mbar_init(bars.mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_addr_smem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_addr_smem;

  const uint32_t s_kv = sbase + kOffKv;
  const uint32_t s_q = sbase + kOffQ;
  const uint32_t s_scale = sbase + kOffScale;
  const uint32_t s_w = sbase + kOffW;
  const float* scale_sm = reinterpret_cast<const float*>(smem + kOffScale);
  const float* w_sm = reinterpret_cast<const float*>(smem + kOffW);

  Walk walk;
  walk.start(grs, gus, p.ctx, G, T, u0, u1);

  if (warp == 0) {
    // =================================================== TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_kv);
      const uint64_t pol_stream = policy_evict_first();  // K pages are read once
      const uint64_t pol_keep = policy_evict_last();      // q and weights
      int it = 0, nq = 0, nw = 0;  // K tiles, Q groups and weight groups issued
      bool ok = true;
      while (ok && walk.next()) {
        const int r0 = walk.r0, n = walk.n;
        ok = wait_or_abort(bars.q_empty, (nq & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(bars.q_full, static_cast<uint32_t>(n * kQRowBytes));
        for (int r = 0; r < n; ++r)
          tma_load_2d(s_q + r * kQRowBytes, &tm_q, 0, (r0 + r) * kHeads, bars.q_full, pol_keep);
        ++nq;
        const int wb = nw & 1;
        ok = wait_or_abort(bars.we(wb), ((nw >> 1) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(bars.wf(wb), static_cast<uint32_t>(n * kHeads * 4));
        bulk_load(s_w + wb * kWBufFloats * 4, p.weights + static_cast<int64_t>(r0) * kHeads,
                  n * kHeads * 4, bars.wf(wb), pol_keep);
        ++nw;
        const int32_t* bt_row = p.block_table + static_cast<int64_t>(r0 + n - 1) * p.bt_stride;
        for (int j = walk.j0; j < walk.j1; ++j, ++it) {
          const int st = it % kStages;
          ok = wait_or_abort(bars.kve(st), ((it / kStages) & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          int32_t blk[2];
          uint32_t bytes = 0;
          for (int h = 0; h < 2; ++h) {
            const int pg = 2 * j + h;
            blk[h] = -1;
            if (pg < walk.npages) {
              int32_t b = (pg < p.bt_stride) ? bt_row[pg] : -1;
              if (b < 0 || b >= p.num_pages) {
                report(p.status, kErrBadBlock);
                b = 0;
              }
              blk[h] = b;
              bytes += kPageValBytesFp8 + kPageTokens * 4;
            }
          }
          mbar_arrive_expect_tx(bars.kvf(st), bytes);
          for (int h = 0; h < 2; ++h) {
            if (blk[h] < 0) continue;
            tma_load_3d(s_kv + st * kKvStageBytes + h * kPageValBytesFp8, &tm_kv, 0, 0, blk[h],
                        bars.kvf(st), pol_stream);
            bulk_load(s_scale + (st * kScaleStageFloats + h * kPageTokens) * 4,
                      p.kv_cache + static_cast<int64_t>(blk[h]) * p.page_stride + kPageValBytesFp8,
                      kPageTokens * 4, bars.kvf(st), pol_stream);
          }
        }
      }
      // Drain: every copy this CTA issued has landed before it may exit (a
      // phase that already completed returns at once).
      for (int i = max(0, it - kStages); i < it; ++i) wait_drain(bars.kvf(i % kStages), (i / kStages) & 1);
      if (nq > 0) wait_drain(bars.q_full, (nq - 1) & 1);
      if (nw > 0) wait_drain(bars.wf((nw - 1) & 1), ((nw - 1) >> 1) & 1);
    }
  } else if (warp == 1) {
    // =================================================== MMA issuer
    if (lane == 0) {
      int it = 0, gi = 0, sc = 0;
      bool ok = true;
      while (ok && walk.next()) {
        const int n = walk.n;
        ok = wait_or_abort(bars.q_full, gi & 1, abort_flag, p.status);
        if (!ok) break;
        for (int j = walk.j0; j < walk.j1 && ok; ++j, ++it) {
          const int st = it % kStages;
          ok = wait_or_abort(bars.kvf(st), (it / kStages) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_tile = s_kv + st * kKvStageBytes;
          int r = 0;
          while (r < n) {
            const int c = sc % kSlots;
            const int len = min(min(n - r, kMaxRowsPerMma), kSlots - c);
            for (int i = 0; i < len && ok; ++i)
              ok = wait_or_abort(bars.te(c + i), (((sc + i) / kSlots) & 1) ^ 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(c * kSlotCols);
            const uint32_t id = idesc(kFmtE4M3, kFmtE4M3, 128, static_cast<uint32_t>(kSlotCols * len));
#pragma unroll
            for (int kk = 0; kk < kHeadDim / 32; ++kk) {
              const uint64_t ad = sdesc_k_sw128(a_tile + kk * 32);
              const uint64_t bd = sdesc_k_sw128(s_q + r * kQRowBytes + kk * 32);
              mma_f8f6f4(d_tmem, ad, bd, id, kk > 0 ? 1u : 0u);
            }
            for (int i = 0; i < len; ++i) mma_commit(bars.tf(c + i));
            r += len;
            sc += len;
          }
          if (!ok) break;
          mma_commit(bars.kve(st));
        }
        if (!ok) break;
        mma_commit(bars.q_empty);
        ++gi;
      }
      // No MMA may still be writing TMEM when it is freed.
      mma_commit(bars.mma_done);
      wait_drain(bars.mma_done, 0);
    }
  } else if (warp >= 4) {
    // =================================================== epilogue
    const int wg = (warp - 4) >> 2;  // warpgroup 0 drains even TMEM slots, 1 odd slots
    const int quarter = warp & 3;    // TMEM lanes this warp may read
    const int tok = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* out_f = static_cast<float*>(p.logits);
    __nv_bfloat16* out_h = static_cast<__nv_bfloat16*>(p.logits);
    int it = 0, gi = 0, sc = 0;
    bool ok = true;
    while (ok && walk.next()) {
      const int r0 = walk.r0, n = walk.n;
      const int wb = gi & 1;
      ok = warp_wait(bars.wf(wb), (gi >> 1) & 1, abort_flag, p.status);
      if (!ok) break;
      const int64_t store_lim = min(static_cast<int64_t>(walk.npages) * kPageTokens, p.logits_stride);
      for (int j = walk.j0; j < walk.j1; ++j, ++it, sc += n) {
        const int st = it % kStages;
        ok = warp_wait(bars.kvf(st), (it / kStages) & 1, abort_flag, p.status);
        if (!ok) break;
        const float kscale = scale_sm[st * kScaleStageFloats + tok];
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.kve(st));
        const int64_t s = static_cast<int64_t>(j) * kTileTokens + tok;
        for (int r = 0; r < n; ++r) {
          const int slot_abs = sc + r;
          if ((slot_abs & 1) != wg) continue;  // each TMEM slot always drains to one warpgroup
          const int slot = slot_abs % kSlots;
          ok = warp_wait(bars.tf(slot), (slot_abs / kSlots) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          uint32_t v[64];
          tmem_ld_x64(t_lane + static_cast<uint32_t>(slot * kSlotCols), v);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.te(slot));
          const float* wr = w_sm + wb * kWBufFloats + r * kHeads;
          float a0 = 0.f, b0 = 0.f, a1 = 0.f, b1 = 0.f, a2 = 0.f, b2 = 0.f, a3 = 0.f, b3 = 0.f;
#pragma unroll
          for (int h = 0; h < kHeads; h += 8) {
            const float4 wa = *reinterpret_cast<const float4*>(wr + h);
            const float4 wc = *reinterpret_cast<const float4*>(wr + h + 4);
            ffma2(a0, b0, relu_f(v[h + 0]), relu_f(v[h + 1]), wa.x, wa.y);
            ffma2(a1, b1, relu_f(v[h + 2]), relu_f(v[h + 3]), wa.z, wa.w);
            ffma2(a2, b2, relu_f(v[h + 4]), relu_f(v[h + 5]), wc.x, wc.y);
            ffma2(a3, b3, relu_f(v[h + 6]), relu_f(v[h + 7]), wc.z, wc.w);
          }
          const float acc = ((a0 + b0) + (a1 + b1)) + ((a2 + b2) + (a3 + b3));
          const int L = p.ctx[r0 + r];
          const float logit = (s < L) ? kscale * acc : -INFINITY;
          if (s < store_lim) {
            const int64_t off = static_cast<int64_t>(r0 + r) * p.logits_stride + s;
            if (p.logits_bf16) out_h[off] = __float2bfloat16_rn(logit);
            else out_f[off] = logit;
          }
        }
        if (!ok) break;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.we(wb));
      ++gi;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_logits_fp8(const LogitsArgs& a, cudaStream_t stream) {
  alignas(64) CUtensorMap tm_q, tm_kv;
  const uint64_t qdims[2] = {static_cast<uint64_t>(kHeadDim),
                             static_cast<uint64_t>(a.num_rows) * kHeads};
  const uint64_t qstrides[1] = {static_cast<uint64_t>(kHeadDim)};
  const uint32_t qbox[2] = {static_cast<uint32_t>(kHeadDim), static_cast<uint32_t>(kHeads)};
  if (!encode_tensor_map_u8(&tm_q, 2, const_cast<uint8_t*>(a.q), qdims, qstrides, qbox, true))
    return cudaErrorInvalidValue;
  const uint64_t kdims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(kPageTokens),
                             static_cast<uint64_t>(a.num_pages)};
  const uint64_t kstrides[2] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(a.page_stride)};
  const uint32_t kbox[3] = {static_cast<uint32_t>(kHeadDim), static_cast<uint32_t>(kPageTokens), 1};
  if (!encode_tensor_map_u8(&tm_kv, 3, const_cast<uint8_t*>(a.kv_cache), kdims, kstrides, kbox, true))
    return cudaErrorInvalidValue;
  Params p;
  p.kv_cache = a.kv_cache;
  p.page_stride = a.page_stride;
  p.num_pages = a.num_pages;
  p.weights = a.weights;
  p.ctx = a.context_lens;
  p.block_table = a.block_table;
  p.bt_stride = a.bt_stride;
  p.indices = a.indices;
  p.schedule = a.schedule;
  p.num_sms = a.num_sms;
  p.logits = a.logits;
  p.logits_bf16 = a.logits_dtype == DSA_LOGITS_BF16 ? 1 : 0;
  p.logits_stride = a.logits_stride;
  p.num_rows = a.num_rows;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(logits_kernel<DSA_KV_FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  logits_kernel<DSA_KV_FP8><<<a.num_sms, kThreads, kSmemBytes, stream>>>(tm_q, tm_kv, p);
  return cudaGetLastError();
}

}  // namespace dsa

namespace dsa {
// FP4-key variant: not built yet.
cudaError_t launch_logits_fp4(const LogitsArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace dsa
