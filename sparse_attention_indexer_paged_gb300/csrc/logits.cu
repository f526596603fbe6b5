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
// The contraction is laid out with the keys as M: for a tile and one row r
// of the group, D[token, h] = sum_d K[token, d] * Q[r, h, d] is a 128 x 64
// tcgen05 MMA (A = the K tile, B = Q row r, K = 128 in steps).  TMEM
// lane = token, so the head-weighted ReLU reduction of a (tile, row) pair
// runs inside one thread with no cross-lane traffic, and a warp's 32 logits
// are 32 consecutive columns.  Per key format:
//   FP8    e4m3 x e4m3, kind::f8f6f4, four K = 32 steps; the fp32 key scale
//          in the epilogue.
//   MXFP4  packed e2m1 x e2m1 with ue8m0 scales per 32 elements on both
//          sides, kind::mxf4 block-scaled, two K = 64 steps; the scales go
//          to TMEM (tcgen05.cp) and the tensor core applies them.
//   FP4    e2m1 keys (e4m3 scales per 16, fp32 per token) against e4m3 q:
//          dequantised to f16 tiles by six warps, kind::f16, eight K = 16 steps.
//
// The CTA's (tile, row) pairs form one stream: pair p goes to TMEM slot
// p mod kSlots (64 columns each; 8 slots, 7 for MXFP4) and is drained by
// epilogue warpgroup p mod 4.  A
// tile's consecutive pairs go out as few MMAs of N = 64 x pairs as the slot
// ring allows (N <= 256, cut where the ring wraps); each chunk waits only for
// its own slots, released by the warpgroups that read their previous pairs,
// and one commit per tile tells the epilogue that all its pairs are in TMEM.
// FP8 calls with full 8-row groups (prefill rows on their request's table),
// whose tiles fill every slot, also commit each earlier chunk of a tile, so
// that its pairs are read while the tile's last chunk waits for slots (on
// decode batches that bookkeeping costs more than it gains).
//
// Rings: K tiles (kStages, released by the tile's MMA commit) and, for FP8
// and MXFP4, the tiles' key scales, which the K producer copies beside the
// values on the same barrier into a ring of kScaleStages tiles (FP8: read by
// the epilogue once the tile's commit has fired; MXFP4: copied to TMEM
// before the tile's MMAs).
//
// Warp roles (FP8 and MXFP4: 640 threads; FP4: 768):
//   warp 0      K producer: per tile the two K pages (3-D tensor map over the
//               pool, page id from the block table) and their key scales
//               (FP4: whole pages by bulk copy); runs ahead across groups.
//   warp 1      MMA issuer and TMEM owner (512 columns): the whole warp walks
//               the work with warp-uniform values; one elected lane issues.
//               For FP8 and MXFP4 keys it also loads each pass's Q rows once
//               the previous pass's MMAs have completed.
//   warp 2      per group: head weights and causal limits (double buffered).
//   warp 3      FP8: no role.  MXFP4: puts the q and key scales in the layout
//               the TMEM copy wants.  FP4: one of six dequantising warps
//               (2, 3, 20-23) that turn raw pages into f16 K tiles.
//   warps 4-19  four epilogue warpgroups: tcgen05.ld of a pair, relu,
//               packed-fp32 FMA with the head weights, key scale, causal
//               mask, store.  Each warp visits only its own pairs.
//
// A wait on an mbarrier that has already completed still costs the waiting
// warp a few hundred cycles; with FP8 and MXFP4 keys most of the MMA warp's
// waits find their phase complete, so it tests each barrier without
// blocking first.
// Every wait is bounded (a CTA abort flag and DSA_ERR_TIMEOUT after 2 s).
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace dsa {
namespace {

// Warps 0-3 have the producer, MMA and loader roles; warps 4-19 are four
// epilogue warpgroups.  FP8 and MXFP4: 20 warps; FP4: plus warps 20-23 so
// that six warps (3, 2, 20-23) share the dequantisation.  Every format reads
// a pair from TMEM in two 32-column pieces (one 64-column load measured 1.3
// us slower on varlen and 2.7 us on MTP; five or six epilogue warpgroups, so
// that a 6-row tile's pairs are read at once, measured slower).
template <int kFmt> constexpr int kEpiWgOf = 4;
template <int kFmt> constexpr int kThreadsOf = kFmt == DSA_KV_FP4 ? 768 : 640;
constexpr int kFp4Converters = 6;
// 64-column TMEM slots; pair p of the CTA's stream uses slot p mod kSlots.
// MXFP4 keeps the last 64 of the 512 columns for its scale factors: the key
// scales of K stage s at columns 448 + 4 s, the q scales of pass row r at
// 480 + 2 r (two rows per 4-column block).
template <int kFmt> constexpr int kSlotsOf = kFmt == DSA_KV_MXFP4 ? 7 : 8;
constexpr int kMaxSlots = 8;
constexpr uint32_t kMxSfaCol = 448;
constexpr uint32_t kMxSfbCol = 480;
constexpr int kTileRing = 8;  // tiles whose "pairs in TMEM" barrier phases are tracked at once
// Full-group FP8 calls (kChunkCommits): every chunk of a tile but its last
// signals its pairs on a ring of chunk barriers (a chunk's MMAs wait for
// slots that pairs at most kSlots positions earlier held, so fewer than 16
// chunks are ever pending)
constexpr int kChunkRing = 16;
constexpr int kScaleStages = 16;   // key scale ring
constexpr int kTmemCols = 512;
constexpr int kPairCols = 64;      // 64 heads of one pair
constexpr int kWBufFloats = kGroupMaxRows * kHeads;       // 512
constexpr int kPageValBytesFp8 = kPageTokens * kHeadDim;  // 8192
constexpr int kFp4PageBytes = DSA_FP4_PAGE_BYTES;         // 4864: values, block scales, token scales
constexpr int kFp4GScaleOffset = kPageTokens * (kHeadDim / 2 + kHeadDim / 16);  // 4608
constexpr int kMxPageValBytes = kPageTokens * (kHeadDim / 2);  // 4096: packed e2m1 values, then 4 ue8m0 scales a token
constexpr int kScaleStageFloats = kTileTokens;            // 128 key scales (or scale words) per tile
constexpr int kMaxKStages = 8;
constexpr int kMaxRawStages = 8;
constexpr int kFp4RawStages = 8;
// q rows per MMA pass over a tile.  FP4: the f16 q of a pass and the raw
// page ring share shared memory (4 rows).  MXFP4: a tile's pairs take
// distinct TMEM slots (7 of them), so groups are walked in passes of 6 rows.
template <int kFmt> constexpr int kPassRowsOf = kFmt == DSA_KV_MXFP4 ? 6 : 4;

// Shared memory layouts (offsets from a 1024-aligned base).
//   FP8:   K ring of e4m3 tiles [128 tokens][128 B] filled by TMA, Q rows e4m3;
//          K-major with the 128-byte swizzle.
//   MXFP4: K ring of packed e2m1 tiles [128 tokens][64 B] filled by TMA, Q
//          rows packed e2m1 [64 heads][64 B]; K-major with the 64-byte
//          swizzle; the pass's q scales in the TMEM copy layout (512 B a row pair).
//   FP4:   raw page pairs (bulk copies of whole pages), dequantised f16 K tiles
//          [2 k-halves][128 tokens][128 B], Q rows in f16 [2 k-halves][pass rows x 64 heads][128 B];
//          K-major with the 128-byte swizzle.
template <int kFmt> struct Lay;
template <> struct Lay<DSA_KV_FP8> {
  static constexpr int kKStages = 8;
  static constexpr int kKStageBytes = 2 * kPageValBytesFp8;  // 16384
  static constexpr int kRawStages = 0;
  static constexpr int kRawStageBytes = 0;
  static constexpr int kQRowBytes = kHeads * kHeadDim;        // 8192
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kKStages * kKStageBytes;
  static constexpr int kOffQsf = kOffQ + kGroupMaxRows * kQRowBytes;  // (unused)
  static constexpr int kOffRaw = kOffQsf;
};
template <> struct Lay<DSA_KV_MXFP4> {
  static constexpr int kKStages = 8;
  static constexpr int kKStageBytes = 2 * kMxPageValBytes;   // 8192
  static constexpr int kRawStages = 0;
  static constexpr int kRawStageBytes = 0;
  static constexpr int kQRowBytes = kHeads * (kHeadDim / 2);  // 4096
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + kKStages * kKStageBytes;
  static constexpr int kOffQsf = kOffQ + kPassRowsOf<DSA_KV_MXFP4> * kQRowBytes;
  static constexpr int kOffRaw = kOffQsf + (kPassRowsOf<DSA_KV_MXFP4> + 1) / 2 * 512;
};
template <> struct Lay<DSA_KV_FP4> {
  static constexpr int kKStages = 2;
  static constexpr int kKStageBytes = 2 * kTileTokens * 128;  // 32768
  static constexpr int kRawStages = kFp4RawStages;
  static constexpr int kRawStageBytes = 2 * kFp4PageBytes;    // 9728
  static constexpr int kQHalfBytes = kPassRowsOf<DSA_KV_FP4> * kHeads * 128;  // one k-half of the pass's f16 q
  static constexpr int kOffQ = 0;
  static constexpr int kOffKv = kOffQ + 2 * kQHalfBytes;
  static constexpr int kOffRaw = kOffKv + kKStages * kKStageBytes;
};
template <int kFmt> struct Smem : Lay<kFmt> {
  using B = Lay<kFmt>;
  static constexpr int kOffScale = B::kOffRaw + B::kRawStages * B::kRawStageBytes;
  static constexpr int kOffW = kOffScale + kScaleStages * kScaleStageFloats * 4;
  static constexpr int kOffCtx = kOffW + 2 * kWBufFloats * 4;  // causal limits of the group's rows
  static constexpr int kOffBar = kOffCtx + 2 * kGroupMaxRows * 4;
  // barriers: kv_full[8], kv_empty[8], raw_full[2], raw_empty[2], q_full, q_empty,
  // w_full[2], w_empty[2], tm_empty[8], mma_done, tile_ready[8], chunk_ready[16]
  static constexpr int kNumBars = 2 * kMaxKStages + 2 * kMaxRawStages + 2 + 4 + kMaxSlots + 1 + kTileRing + kChunkRing;
  static constexpr int kOffTmemAddr = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemAddr + 4;
  static constexpr int kOffWalk = kOffAbort + 4;  // WalkRanges
  static constexpr int kBytes = kOffWalk + 6 * 4 + 1024;  // + alignment slack
  static_assert(B::kOffQ % 1024 == 0 && B::kOffKv % 1024 == 0 && B::kKStageBytes % 1024 == 0,
                "MMA tiles need 1024-byte alignment");
  static_assert(B::kOffRaw % 16 == 0 && B::kRawStageBytes % 16 == 0, "bulk copies need 16 bytes");
  static_assert((B::kKStages & (B::kKStages - 1)) == 0 && B::kKStages <= kMaxKStages, "K ring");
  static_assert(kOffScale % 512 == 0, "scale blocks are copied to TMEM from 16-byte rows");
  static_assert(kOffBar % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kBytes <= 232448, "over the per-CTA shared memory limit");
};
static_assert(kSlotsOf<DSA_KV_FP8> * kPairCols == kTmemCols && kSlotsOf<DSA_KV_FP4> * kPairCols == kTmemCols &&
                  kSlotsOf<DSA_KV_MXFP4> * kPairCols == kMxSfaCol &&
                  kMxSfaCol + 4 * Lay<DSA_KV_MXFP4>::kKStages <= kMxSfbCol &&
                  kMxSfbCol + 4 * ((kPassRowsOf<DSA_KV_MXFP4> + 1) / 2) <= kTmemCols,
              "TMEM slots and the MXFP4 scale columns");
static_assert(kGroupMaxRows <= kSlotsOf<DSA_KV_FP8> && kPassRowsOf<DSA_KV_MXFP4> <= kSlotsOf<DSA_KV_MXFP4> &&
                  kPassRowsOf<DSA_KV_FP4> <= kSlotsOf<DSA_KV_FP4> && kSlotsOf<DSA_KV_FP8> <= kMaxSlots,
              "a tile's pairs take distinct TMEM slots");
static_assert(group_rows_for(DSA_KV_FP4) == kPassRowsOf<DSA_KV_FP4> &&
                  group_rows_for(DSA_KV_MXFP4) == kPassRowsOf<DSA_KV_MXFP4>,
              "the schedule's groups of the FP4 formats are one row pass each");
static_assert(Lay<DSA_KV_FP8>::kKStages == kTileRing && Lay<DSA_KV_MXFP4>::kKStages == kTileRing,
              "FP8 and MXFP4 tiles signal their pairs on the K stage's own barrier");
static_assert(Lay<DSA_KV_MXFP4>::kKStages <= kMaxRawStages, "MXFP4 scale barriers reuse the raw ring's");
static_assert(kScaleStageFloats * 4 == 512, "a tile's key scales are one 512-byte TMEM copy block (MXFP4)");
static_assert(kFp4AHalfLo == (kTileTokens * 128) >> 4, "f16 K operand halves as laid out by the dequantising warps");
static_assert(kFp4RawStages <= kMaxRawStages, "raw stages");

struct Params {
  const uint8_t* q;
  const uint8_t* q_scale;  // MXFP4: ue8m0 [T][H][D/32]
  const uint8_t* kv_cache;
  int64_t page_stride;
  int64_t num_pages;
  const float* weights;
  const int32_t* ctx;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* bt_rows;  // block-table row of each row (null: the row itself)
  int32_t bt_num_rows;     // rows of the block table when bt_rows is set
  const int32_t* indices;
  const int32_t* schedule;
  int32_t num_sms;
  void* logits;
  int64_t logits_stride;
  int32_t num_rows;
  int32_t* status;
};

// The block-table row that row `row` reads its pages from: the row itself,
// or, with a per-row map (prefill rows reading their request's table), the
// mapped row; a mapped row outside the table is reported and row 0 read.
__device__ __forceinline__ const int32_t* table_row(const Params& p, int row) {
  int64_t tr = row;
  if (p.bt_rows != nullptr) {
    tr = __ldg(p.bt_rows + row);
    if (tr < 0 || tr >= p.bt_num_rows) {
      report(p.status, kErrBadBlock);
      tr = 0;
    }
  }
  return p.block_table + tr * p.bt_stride;
}

struct Bars {
  uint32_t kv_full, kv_empty, raw_full, raw_empty, q_full, q_empty, w_full,
      w_empty, tm_empty, mma_done, tile_ready, chunk_ready;
  __device__ uint32_t kvf(int s) const { return kv_full + 8 * s; }
  __device__ uint32_t kve(int s) const { return kv_empty + 8 * s; }
  __device__ uint32_t rwf(int s) const { return raw_full + 8 * s; }
  __device__ uint32_t rwe(int s) const { return raw_empty + 8 * s; }
  // MXFP4 (no raw ring): K stage s's key scales are in the TMEM copy layout
  __device__ uint32_t sfr(int s) const { return raw_full + 8 * s; }
  __device__ uint32_t wf(int b) const { return w_full + 8 * b; }
  __device__ uint32_t we(int b) const { return w_empty + 8 * b; }
  // TMEM slot s: drained by the warpgroup of the pair in it
  // Tile i's pairs are in TMEM: one MMA commit per tile.  With 8 K stages
  // (FP8, MXFP4) this is the stage's kv_empty barrier; FP4 has 2 stages and a
  // ring of its own, so that a warp waiting for tile i never finds the
  // barrier already two phases on.
  __device__ uint32_t tr(uint32_t i, bool own_ring) const {
    return own_ring ? tile_ready + 8 * (i & (kTileRing - 1)) : kv_empty + 8 * (i & (kTileRing - 1));
  }
  __device__ uint32_t te(uint32_t s) const { return tm_empty + 8 * s; }
  // chunk c of the CTA's early chunks (all but each tile's last) has its
  // pairs in TMEM
  __device__ uint32_t ch(uint32_t c) const { return chunk_ready + 8 * (c & (kChunkRing - 1)); }
};

// The CTA's walk over its units: two ranges of the schedule's sorted unit
// sequence (one from each end, the heavy one first), and within them the
// groups in sorted order with the tiles [j0, j1) of each group that belong
// to this CTA.  A group of n rows is walked as ceil(n / kPassRows) row passes
// over the same tiles (one pass when kPassRows = 8; the FP4 path uses passes
// of 4 rows so that its f16 copy of the q rows fits next to a deep page
// ring).  Every role runs the
// same walk with all 32 lanes of its warp: the lanes search the unit starts
// 32 entries at a time and read a group's causal limits in parallel.  The
// schedule arrays are found from the kernel parameters on each call, so the
// walk keeps no pointers in registers.
// This CTA's two unit ranges and the sorted position where each starts,
// resolved once per CTA (warp 0, before the roles start) into shared memory.
struct WalkRanges {
  int32_t u0[2], u1[2], k0[2];
};

// this CTA's units: [a0, a1) from the light end, [b0, b1) from the heavy end
__device__ __forceinline__ void cta_ranges(const int32_t* sched, int S, int T, int& a0, int& a1, int& b0, int& b1) {
  const SchedLayout L(S, T);
  const int U = sched[5];
  a0 = min(max(sched[L.left + blockIdx.x], 0), U);
  a1 = min(max(sched[L.left + blockIdx.x + 1], a0), U);
  b1 = min(max(sched[L.right + blockIdx.x], a1), U);
  b0 = min(max(sched[L.right + blockIdx.x + 1], a1), b1);
}

// The largest sorted position k in [0, G) with sus[k] <= u (sus is
// non-decreasing, sus[0] = 0), by the whole warp: each round narrows
// [lo, hi) 32-fold.
__device__ __forceinline__ int seek_position(const int32_t* sus, int G, int u, int lane) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + lane * step;
    const bool le = idx < hi && __ldg(sus + idx) <= u;
    const uint32_t m = __ballot_sync(0xffffffffu, le);
    lo += (31 - __clz(m | 1u)) * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

template <int kPassRows>
struct Walk {
  int G, k, u, u_end, range;
  int g_r0, g_n, pass, npass;  // current group and row pass
  // current pass: rows [r0, r0 + n) of the group's tiles [j0, j1)
  int r0, n, npages, j0, j1;
  int32_t lane_ctx;  // causal limit of row r0 + lane (lanes below n)

  __device__ void start(const int32_t* sched, const WalkRanges* wr) {
    G = sched[4];
    range = 0;
    u = wr->u0[0];
    u_end = wr->u1[0];
    k = wr->k0[0];
    pass = npass = 0;
  }

  // Loads the next row pass that holds units of this CTA; false when done.
  __device__ bool next(const int32_t* sched, int S, int T, const int32_t* ctx, const WalkRanges* wr, int lane) {
    constexpr bool kOnePass = kPassRows >= kGroupMaxRows;  // every group in one pass
    if (!kOnePass && pass + 1 < npass) {
      ++pass;  // same group and tiles, next rows
    } else {
      const SchedLayout L(S, T);
      const int32_t* sus = sched + L.sus;
      while (u < u_end && k < G && __ldg(sus + k + 1) <= u) ++k;
      if (u >= u_end || k >= G) {
        if (range != 0) return false;
        range = 1;  // on to the second range
        u = wr->u0[1];
        u_end = wr->u1[1];
        k = wr->k0[1];
        while (u < u_end && k < G && __ldg(sus + k + 1) <= u) ++k;
        if (u >= u_end || k >= G) return false;
      }
      const int s0 = __ldg(sus + k), s1 = __ldg(sus + k + 1);
      const int32_t w = __ldg(sched + L.pos + k);
      g_r0 = w & kPosRowMask;
      g_n = static_cast<int>(static_cast<uint32_t>(w) >> kPosRowsShift);
      if (g_n <= 0 || g_n > kGroupMaxRows || g_r0 + g_n > T) return false;
      int lmax = lane < g_n ? __ldg(ctx + g_r0 + lane) : 0;
#pragma unroll
      for (int o = 4; o; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));  // lanes 0..7
      lmax = __shfl_sync(0xffffffffu, lmax, 0);
      npages = (lmax + kPageTokens - 1) / kPageTokens;  // of the whole group: every pass writes its columns
      j0 = u - s0;
      j1 = min(s1, u_end) - s0;
      u = s0 + j1;
      pass = 0;
      npass = kOnePass ? 1 : (g_n + kPassRows - 1) / kPassRows;
    }
    r0 = kOnePass ? g_r0 : g_r0 + pass * kPassRows;
    n = kOnePass ? g_n : min(g_n - pass * kPassRows, kPassRows);
    lane_ctx = lane < n ? __ldg(ctx + r0 + lane) : 0;
    return true;
  }
};

// Wait by every lane of a warp: each lane's own acquire orders its later
// reads after the completed phase; the vote keeps the warp's control flow
// uniform (false on timeout or abort).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag, status));
}

// The chunk of a tile's pairs that starts at stream position pos with
// `left` pairs to go: contiguous TMEM slots (cut where the slot ring wraps),
// at most 4 pairs (N <= 256).  The MMA warp issues, and the epilogue waits
// for, the same chunks.
template <int kSlots>
__device__ __forceinline__ uint32_t chunk_len(uint32_t pos, uint32_t left) {
  return min(min(left, static_cast<uint32_t>(kSlots) - pos % kSlots), 4u);
}

__device__ __forceinline__ void store_logit(float* dst, float v) { *dst = v; }
__device__ __forceinline__ void store_logit(__nv_bfloat16* dst, float v) { *dst = __float2bfloat16_rn(v); }

template <int kFmt, typename OutT, bool kChunkCommits>
__global__ void __launch_bounds__(kThreadsOf<kFmt>, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                  const Params p) {
  using L = Smem<kFmt>;
  constexpr bool kDq = kFmt == DSA_KV_FP4;    // dequantising pipeline: FP4 keys
  constexpr bool kMx = kFmt == DSA_KV_MXFP4;  // block-scaled e2m1 MMA: MXFP4 keys and q
  constexpr int kSlots = kSlotsOf<kFmt>;
  constexpr int kEpiWg = kEpiWgOf<kFmt>;
  constexpr int kEpiWarps = 4 * kEpiWg;
  constexpr int kStages = L::kKStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The schedule (and everything else an earlier kernel on the stream wrote)
  // is read only once that kernel has finished; the kernel after this one
  // (the top-k) may be scheduled as this one's CTAs leave their SMs.
  grid_dep_wait();
  grid_dep_launch();
  // ---- the schedule must be the one built for these rows, mode and SM count
  const int32_t* sched = p.schedule;
  const int S = p.num_sms;
  const int T = p.num_rows;
  if (sched[0] != kScheduleMagic || sched[1] != T || sched[2] != (p.indices != nullptr ? 1 : 0) ||
      sched[3] != S || sched[6] != kTileTokens || sched[7] < 1 || sched[7] > kGroupMaxRows ||
      static_cast<int>(gridDim.x) != S || sched[4] < 0 || sched[4] > T || sched[5] < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(p.status, kErrScheduleMismatch);
    return;
  }
  {
    int a0, a1, b0, b1;
    cta_ranges(sched, S, T, a0, a1, b0, b1);
    if ((a0 >= a1 && b0 >= b1) || sched[4] == 0) return;  // no work: the whole CTA leaves before any set-up
  }

  Bars bars;
  bars.kv_full = sbase + L::kOffBar;
  bars.kv_empty = bars.kv_full + 8 * kMaxKStages;
  bars.raw_full = bars.kv_empty + 8 * kMaxKStages;
  bars.raw_empty = bars.raw_full + 8 * kMaxRawStages;
  bars.q_full = bars.raw_empty + 8 * kMaxRawStages;
  bars.q_empty = bars.q_full + 8;
  bars.w_full = bars.q_empty + 8;
  bars.w_empty = bars.w_full + 16;
  bars.tm_empty = bars.w_empty + 16;
  bars.mma_done = bars.tm_empty + 8 * kMaxSlots;
  bars.tile_ready = bars.mma_done + 8;
  bars.chunk_ready = bars.tile_ready + 8 * kTileRing;
  uint32_t* tmem_addr_smem = reinterpret_cast<uint32_t*>(smem + L::kOffTmemAddr);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kOffAbort);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars.kvf(s), kDq ? kFp4Converters : 1);  // TMA (FP8, MXFP4) or the dequantising warps (FP4)
      mbar_init(bars.kve(s), 1);  // the MMA commit of the tile: stage free, the tile's pairs in TMEM
    }
    for (int s = 0; s < L::kRawStages; ++s) {
      mbar_init(bars.rwf(s), 1);
      mbar_init(bars.rwe(s), kFp4Converters);  // the dequantising warps
    }
    if (kMx)
      for (int s = 0; s < kStages; ++s) mbar_init(bars.sfr(s), 1);  // the scale warp
    // the MMA warp's TMA (FP8), plus the scale warp's q scales (MXFP4), or
    // the converting warps (FP4)
    mbar_init(bars.q_full, kDq ? kFp4Converters : (kMx ? 2 : 1));
    mbar_init(bars.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.wf(b), 1);
      mbar_init(bars.we(b), kEpiWarps);
    }
    for (uint32_t sl = 0; sl < kSlots; ++sl)
      mbar_init(bars.te(sl), 4);  // the four warps of the pair's warpgroup have read it
    mbar_init(bars.mma_done, 1);
    for (int i = 0; i < kTileRing; ++i) mbar_init(bars.tile_ready + 8 * i, 1);  // the tile's MMA commit
    for (int i = 0; i < kChunkRing; ++i) mbar_init(bars.chunk_ready + 8 * i, 1);  // a chunk's MMA commit
    *abort_flag = 0;
    fence_mbar_init();
  }
  WalkRanges* walk_ranges = reinterpret_cast<WalkRanges*>(smem + L::kOffWalk);
  if (warp == 0) {
    int a0, a1, b0, b1;
    cta_ranges(sched, S, T, a0, a1, b0, b1);
    const int32_t* sus = sched + SchedLayout(S, T).sus;
    const int ka = seek_position(sus, sched[4], a0, lane);
    const int kb = seek_position(sus, sched[4], b0, lane);
    // the heavy (right, many-row) range first: a CTA that ends on light
    // tiles drains faster than one that ends on a chain of many-row tiles
    // (measured faster for every key format)
    if (lane == 0) *walk_ranges = WalkRanges{{b0, a0}, {b1, a1}, {kb, ka}};
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_addr_smem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_addr_smem;

  const uint32_t s_kv = sbase + L::kOffKv;
  const uint32_t s_q = sbase + L::kOffQ;
  const uint32_t s_scale = sbase + L::kOffScale;
  const uint32_t s_w = sbase + L::kOffW;
  float* scale_sm = reinterpret_cast<float*>(smem + L::kOffScale);
  const float* w_sm = reinterpret_cast<const float*>(smem + L::kOffW);
  int32_t* ctx_sm = reinterpret_cast<int32_t*>(smem + L::kOffCtx);

  Walk<kFmt == DSA_KV_FP8 ? kGroupMaxRows : kPassRowsOf<kFmt>> walk;
  walk.start(sched, walk_ranges);

  // =================================================== FP4 dequantisation (warps 3, 2, 20-23)
  // The six warps share every tile: work item k (0..511) is 32 elements
  // (one 16-byte piece) of token k / 4, and warp `part` takes the items
  // k = 32 * part + lane (mod 192).  e2m1 values times their e4m3 block scale
  // -> f16 (exact: at most 6 significant bits) into the swizzled A-operand
  // tile; token scales into the scale ring.  The warps also share the
  // conversion of every pass's q rows (e4m3 -> f16, exact) into the swizzled
  // B-operand layout.  Warp 2 first loads the pass's head weights and causal
  // limits (double buffered).
  auto fp4_worker = [&]() {
    using LF = Lay<DSA_KV_FP4>;  // (compiled, never run, for the other formats)
    constexpr int kPg = kFp4PageBytes;
    constexpr int kStride = 32 * kFp4Converters;
    const int part = warp == 3 ? 0 : (warp == 2 ? 1 : warp - (4 + kEpiWarps) + 2);
    const uint64_t pol_keep = policy_evict_last();
    const uint32_t q_half = static_cast<uint32_t>(LF::kQHalfBytes);
    int it = 0, nq = 0, nw = 0;
    bool ok = true;
    while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
      const int r0 = walk.r0, n = walk.n;
      if (part == 1) {
        const int wb = nw & 1;
        ok = warp_wait(bars.we(wb), ((nw >> 1) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        if (lane < n) ctx_sm[wb * kGroupMaxRows + lane] = walk.lane_ctx;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bars.wf(wb), static_cast<uint32_t>(n * kHeads * 4));
          bulk_load(s_w + wb * kWBufFloats * 4, p.weights + static_cast<int64_t>(r0) * kHeads,
                    n * kHeads * 4, bars.wf(wb), pol_keep);
        }
        ++nw;
      }
      // q rows of the pass, once the previous pass's MMAs have completed
      ok = warp_wait(bars.q_empty, (nq & 1) ^ 1, abort_flag, p.status);
      if (!ok) break;
      // 8 e4m3 codes per step; the warps take interleaved 32-chunk blocks
      const uint2* qsrc = reinterpret_cast<const uint2*>(p.q + static_cast<int64_t>(r0) * kHeads * kHeadDim);
      const int nchunks = n * kHeads * (kHeadDim / 8);
      for (int i = part * 32 + lane; i < nchunks; i += kStride) {
        const uint2 c = __ldg(qsrc + i);
        const int R = i >> 4;      // q row (row * 64 + head) within the pass
        const int c16 = i & 15;    // 8-element chunk along d
        uint4 o;
        o.x = e4m3x2_to_f16x2(c.x & 0xffffu);
        o.y = e4m3x2_to_f16x2(c.x >> 16);
        o.z = e4m3x2_to_f16x2(c.y & 0xffffu);
        o.w = e4m3x2_to_f16x2(c.y >> 16);
        const uint32_t off = static_cast<uint32_t>(c16 >> 3) * q_half + static_cast<uint32_t>(R >> 3) * 1024u +
                             static_cast<uint32_t>(R & 7) * 128u + (static_cast<uint32_t>((c16 & 7) ^ (R & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + LF::kOffQ + off) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full);
      ++nq;
      for (int j = walk.j0; j < walk.j1; ++j, ++it) {
        const int rs = it % LF::kRawStages;
        const int st = it % LF::kKStages;
        const int ss = it % kScaleStages;
        ok = warp_wait(bars.rwf(rs), (it / LF::kRawStages) & 1, abort_flag, p.status) &&
             warp_wait(bars.kve(st), ((it / LF::kKStages) & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        const uint8_t* raw = smem + LF::kOffRaw + rs * LF::kRawStageBytes;
        for (int t = part * 32 + lane; t < kTileTokens; t += kStride)  // token scales -> scale ring
          scale_sm[ss * kScaleStageFloats + t] =
              *reinterpret_cast<const float*>(raw + (t >> 6) * kPg + kFp4GScaleOffset + (t & 63) * 4);
        uint8_t* tile = smem + LF::kOffKv + st * LF::kKStageBytes;
#pragma unroll 1
        for (int k = part * 32 + lane; k < kTileTokens * 4; k += kStride) {
          const int tk = k >> 2, q4 = k & 3;  // token within the tile, 32-element piece
          const uint8_t* tokp = raw + (tk >> 6) * kPg;
          const int slot = tk & 63;
          const uint4 pv = *reinterpret_cast<const uint4*>(tokp + slot * (kHeadDim / 2) + q4 * 16);
          // block scales of the piece's two 16-element blocks
          uint32_t sb[2];
          const uint32_t s2 = e4m3x2_to_f16x2(
              *reinterpret_cast<const uint16_t*>(tokp + kPageTokens * (kHeadDim / 2) + slot * 8 + q4 * 2));
          sb[0] = __byte_perm(s2, 0, 0x1010);
          sb[1] = __byte_perm(s2, 0, 0x3232);
          const uint32_t words[4] = {pv.x, pv.y, pv.z, pv.w};
          const uint32_t row = static_cast<uint32_t>(tk >> 3) * 1024u + static_cast<uint32_t>(tk & 7) * 128u;
#pragma unroll
          for (int wv = 0; wv < 4; ++wv) {  // 8 elements per word
            const int c16 = q4 * 4 + wv;     // chunk of elements 8*c16 .. 8*c16+7
            uint32_t h[4];
            e2m1x8_to_f16x2(words[wv], h);
            const uint32_t sc = sb[wv >> 1];
            uint4 o;
            o.x = hmul2_u32(h[0], sc);
            o.y = hmul2_u32(h[1], sc);
            o.z = hmul2_u32(h[2], sc);
            o.w = hmul2_u32(h[3], sc);
            const uint32_t off = static_cast<uint32_t>(c16 >> 3) * (kTileTokens * 128u) + row +
                                 (static_cast<uint32_t>((c16 & 7) ^ (tk & 7)) << 4);
            *reinterpret_cast<uint4*>(tile + off) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bars.rwe(rs));
          mbar_arrive(bars.kvf(st));
        }
      }
    }
    if (part == 1 && lane == 0 && nw > 0) wait_drain(bars.wf((nw - 1) & 1), ((nw - 1) >> 1) & 1);
  };

  if (warp == 0) {
    // =================================================== producer: K pages
    // The whole warp walks the work: block ids are fetched 32 at a time with
    // one coalesced load and handed out by shuffle; lane 0 waits and issues.
    // Nothing here waits on a group boundary, so the ring runs ahead across
    // groups.
    if constexpr (!kDq) {
      if (lane == 0) prefetch_tensormap(&tm_kv);
    }
    const uint64_t pol_stream = policy_evict_first();  // K pages are read once
    constexpr int kRing = kDq ? L::kRawStages : kStages;
    int it = 0;  // tiles issued
    bool ok = true;
    while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
      const int r0 = walk.r0, n = walk.n;
      const int32_t* bt_row = table_row(p, walk.g_r0 + walk.g_n - 1);  // the group's last row
      int32_t lane_blk = -1;  // block id of page (pg_base + lane)
      int pg_base = -32;
      for (int j = walk.j0; j < walk.j1; ++j, ++it) {
        if (2 * j >= pg_base + 32) {
          pg_base = 2 * j;
          const int pg = pg_base + lane;
          lane_blk = -1;
          if (pg < walk.npages) {
            int32_t b = (pg < p.bt_stride) ? __ldg(bt_row + pg) : -1;
            if (b < 0 || b >= p.num_pages) {
              report(p.status, kErrBadBlock);
              b = 0;
            }
            lane_blk = b;
          }
        }
        const int32_t blk0 = __shfl_sync(0xffffffffu, lane_blk, 2 * j - pg_base);
        const int32_t blk1 = __shfl_sync(0xffffffffu, lane_blk, 2 * j + 1 - pg_base);
        if (lane == 0) {
          const int st = it % kRing;
          const uint32_t empty_bar = kDq ? bars.rwe(st) : bars.kve(st);
          const uint32_t full_bar = kDq ? bars.rwf(st) : bars.kvf(st);
          ok = wait_or_abort(empty_bar, ((it / kRing) & 1) ^ 1, abort_flag, p.status);
          if (ok) {
            const int npg = (blk0 >= 0 ? 1 : 0) + (blk1 >= 0 ? 1 : 0);
            if constexpr (kDq) {
              // whole pages: packed values and their scales
              constexpr int kPg = kFp4PageBytes;
              mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(npg * kPg));
              const uint32_t dst = sbase + L::kOffRaw + st * L::kRawStageBytes;
              if (blk0 >= 0)
                bulk_load(dst, p.kv_cache + static_cast<int64_t>(blk0) * p.page_stride, kPg, full_bar,
                          pol_stream);
              if (blk1 >= 0)
                bulk_load(dst + kPg, p.kv_cache + static_cast<int64_t>(blk1) * p.page_stride, kPg, full_bar,
                          pol_stream);
            } else {
              // the two pages' values (tensor map, swizzled) and their key
              // scales (plain copies into the scale ring), one barrier: FP8
              // pages hold 8192 value bytes then an fp32 scale a token, MXFP4
              // pages 4096 packed e2m1 bytes then 4 ue8m0 block scales a token
              constexpr uint32_t kVal = kMx ? kMxPageValBytes : kPageValBytesFp8;
              constexpr uint32_t kSc = kPageTokens * 4;
              const uint32_t sc_dst = s_scale + (it % kScaleStages) * kScaleStageFloats * 4;
              mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(npg) * (kVal + kSc));
              if (blk0 >= 0) {
                tma_load_3d(s_kv + st * L::kKStageBytes, &tm_kv, 0, 0, blk0, full_bar, pol_stream);
                bulk_load(sc_dst, p.kv_cache + static_cast<int64_t>(blk0) * p.page_stride + kVal, kSc, full_bar,
                          pol_stream);
              }
              if (blk1 >= 0) {
                tma_load_3d(s_kv + st * L::kKStageBytes + kVal, &tm_kv, 0, 0, blk1, full_bar, pol_stream);
                bulk_load(sc_dst + kSc, p.kv_cache + static_cast<int64_t>(blk1) * p.page_stride + kVal, kSc,
                          full_bar, pol_stream);
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    // Drain: every copy this CTA issued has landed before it may exit (a
    // phase that already completed returns at once).
    if (lane == 0) {
      for (int i = max(0, it - kRing); i < it; ++i)
        wait_drain(kDq ? bars.rwf(i % kRing) : bars.kvf(i % kRing), (i / kRing) & 1);
    }
  } else if (warp == 2 || warp == 3 || warp >= 4 + kEpiWarps) {
    if constexpr (!kDq) {
      if (warp == 3) {
        // FP8: no role (the K producer brings each tile's key scales with its
        // values); the warp waits at the final barrier.
        if constexpr (kMx) {
          // =================================================== MXFP4: scales into the TMEM copy layout
          // A 128-row scale block goes to TMEM as one copy that gives lane l,
          // column c the source word 4 l + c, and row x's scales must land in
          // lane x mod 32, column x / 32: so row x's word moves from position x
          // to 4 (x mod 32) + x / 32, a 4 x 32 transpose (lane l gathers rows
          // l, 32 + l, 64 + l, 96 + l and stores them as one 16-byte row).
          //   q: per pass, two rows (128 B-operand rows) per block, straight
          //      from global memory, once the previous pass's MMAs (and the
          //      copies before them) have completed; then one arrival on q_full.
          //   keys: per tile, in place in the scale ring once the tile has
          //      landed; then the stage's sfr barrier.
          const uint32_t* qsc = reinterpret_cast<const uint32_t*>(p.q_scale);
          uint8_t* qsf = smem + L::kOffQsf;
          uint32_t it = 0, gi = 0;
          bool ok = true;
          while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
            const int r0 = walk.r0, n = walk.n;
            ok = warp_wait(bars.q_empty, (gi & 1) ^ 1, abort_flag, p.status);
            if (!ok) break;
            for (int b = 0; 2 * b < n; ++b) {
              uint32_t w[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int r = 2 * b + (c >> 1);  // row of the pass; heads 32 (c & 1) + lane
                w[c] = r < n ? __ldg(qsc + static_cast<int64_t>(r0 + r) * kHeads + 32 * (c & 1) + lane)
                             : 0x7f7f7f7fu;
              }
              *reinterpret_cast<uint4*>(qsf + b * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.q_full);
            ++gi;
            for (int j = walk.j0; j < walk.j1; ++j, ++it) {
              const uint32_t st = it & (kStages - 1);
              ok = warp_wait(bars.kvf(st), (it / kStages) & 1, abort_flag, p.status);
              if (!ok) break;
              uint32_t* blk = reinterpret_cast<uint32_t*>(smem + L::kOffScale) +
                              (it & (kScaleStages - 1)) * kScaleStageFloats;
              const uint4 v = make_uint4(blk[lane], blk[32 + lane], blk[64 + lane], blk[96 + lane]);
              __syncwarp();
              *reinterpret_cast<uint4*>(blk + 4 * lane) = v;
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(bars.sfr(st));
            }
          }
        }
      } else {
        // =================================================== per group: weights and causal limits
        // A separate producer: the epilogue may hold a group's weights until TMEM
        // buffers that also carry later groups' pairs complete, so these loads
        // must never sit in front of the Q and K loads.
        const uint64_t pol_keep = policy_evict_last();
        int nw = 0;
        bool ok = true;
        while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
          const int r0 = walk.r0, n = walk.n;
          const int wb = nw & 1;
          ok = warp_wait(bars.we(wb), ((nw >> 1) & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          // lanes below n write their row's causal limit; the fence and the warp
          // barrier order those writes before lane 0's release on wf
          if (lane < n) ctx_sm[wb * kGroupMaxRows + lane] = walk.lane_ctx;
          __threadfence_block();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(bars.wf(wb), static_cast<uint32_t>(n * kHeads * 4));
            bulk_load(s_w + wb * kWBufFloats * 4, p.weights + static_cast<int64_t>(r0) * kHeads,
                      n * kHeads * 4, bars.wf(wb), pol_keep);
          }
          ++nw;
        }
        if (lane == 0 && nw > 0) wait_drain(bars.wf((nw - 1) & 1), ((nw - 1) >> 1) & 1);
      }
    } else {
      fp4_worker();
    }
  } else if (warp == 1) {
    // =================================================== MMA issuer
    // The whole warp walks the work, so every value feeding an MMA is
    // warp-uniform; one elected lane issues the MMAs and commits.  Each MMA
    // occupies the tensor unit for at least ~48 cycles whatever its N, so a
    // tile's rows go out as few wide MMAs as the TMEM buffers allow.
    // instruction descriptor for N = 64 * len: the N field (N >> 3 at bit
    // 17) grows by len << 20; format code 0 is e4m3 for kind::f8f6f4 and f16
    // for kind::f16
    const uint32_t id_base = kMx ? idesc_mxf4(128, 0) : idesc(0, 0, 128, 0);
    constexpr uint32_t kHi = kMx ? kSdescHiSw64 : kSdescHi;
    const uint32_t a_lo0 = sdesc_lo(s_kv), q_lo0 = sdesc_lo(s_q);
    constexpr uint32_t kStageLo = L::kKStageBytes >> 4;
    // one q row (64 heads) of B: 8192 bytes of e4m3 (FP8), 64 f16 rows of
    // 128 bytes in each k-half (FP4), 4096 bytes of packed e2m1 (MXFP4)
    constexpr uint32_t kQRowLo = (kMx ? kHeads * (kHeadDim / 2) : kHeads * 128) >> 4;
    // FP4: the B operand's second k-half follows the pass's first
    constexpr uint32_t kQHalfLo = Lay<DSA_KV_FP4>::kQHalfBytes >> 4;
    const uint32_t issue = elect_one() ? 1u : 0u;
    const bool leader = issue != 0;
    if constexpr (!kDq) {
      if (leader) prefetch_tensormap(&tm_q);
    }
    const uint64_t pol_keep = policy_evict_last();  // q
    uint32_t it = 0, gi = 0, pos = 0, nq = 0, ce = 0;  // tiles, groups, pairs, Q loads, early chunks issued
    bool ok = true;
    while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
      const uint32_t n = static_cast<uint32_t>(walk.n);
      if constexpr (!kDq) {
        // Q buffer free once the previous group's MMAs have completed
        ok = warp_wait(bars.q_empty, (gi & 1) ^ 1, abort_flag, p.status);
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(bars.q_full, n * static_cast<uint32_t>(L::kQRowBytes));
          for (uint32_t r = 0; r < n; ++r)
            tma_load_2d(s_q + r * L::kQRowBytes, &tm_q, 0, (walk.r0 + static_cast<int>(r)) * kHeads,
                        bars.q_full, pol_keep);
        }
        ++nq;
      }
      ok = warp_wait(bars.q_full, gi & 1, abort_flag, p.status);
      if (!ok) break;
      if constexpr (kMx) {
        // the pass's q scales to TMEM: rows 2b, 2b + 1 at columns kMxSfbCol + 4b
        tc_fence_after();
        const uint32_t s_qsf = sbase + L::kOffQsf;
        for (uint32_t b = 0; 2 * b < n; ++b)
          tmem_cp_scales(issue, tmem + kMxSfbCol + 4 * b, sdesc_lo_plain(s_qsf + 512 * b), kSdescHiPlain);
      }
      for (int j = walk.j0; j < walk.j1; ++j, ++it) {
        const uint32_t st = it & (kStages - 1);
        // A wait that finds its phase complete still costs a few hundred
        // cycles.  With FP8 and MXFP4 keys the K stage and most slots are
        // ready when the MMA warp comes to them (the K stream runs ahead), so
        // each barrier is first tested without blocking; FP4 waits at once
        // (its stages and slots are mostly still pending, and a test first
        // only delays the wake-up).  The warp votes once per wait group.
        {
          // MXFP4: the stage's scales are in the copy layout too (the scale
          // warp saw the stage land first)
          const uint32_t kvp = (it / kStages) & 1;
          const uint32_t kb = kMx ? bars.sfr(st) : bars.kvf(st);
          ok = __all_sync(0xffffffffu,
                          (!kDq && mbar_test(kb, kvp)) || wait_or_abort(kb, kvp, abort_flag, p.status));
        }
        if (!ok) break;
        if constexpr (kMx) {
          tc_fence_after();
          tmem_cp_scales(issue, tmem + kMxSfaCol + 4 * st,
                         sdesc_lo_plain(s_scale + (it & (kScaleStages - 1)) * kScaleStageFloats * 4), kSdescHiPlain);
        }
        const uint32_t a_lo = a_lo0 + st * kStageLo;
        uint32_t b_lo = q_lo0;
        uint32_t left = n;
        do {  // the tile's rows, cut where a TMEM buffer ends
          const uint32_t c = pos % kSlots;
          const uint32_t len = chunk_len<kSlots>(pos, left);
          // pair pos + i goes to slot c + i, free once the pair kSlots
          // positions earlier has been read by its warpgroup (a tile's
          // n <= kSlots pairs take n distinct slots); each chunk waits only
          // for its own slots
          bool mine = true;
          for (uint32_t i = 0; i < len && mine; ++i) {
            const uint32_t b = bars.te(c + i), pr = (((pos + i) / kSlots) & 1) ^ 1;
            mine = (!kDq && mbar_test(b, pr)) || wait_or_abort(b, pr, abort_flag, p.status);
          }
          ok = __all_sync(0xffffffffu, mine);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + c * kPairCols;
          if constexpr (kMx)
            mma_mxf4_k128(issue, d_tmem, a_lo, b_lo, kHi, id_base + (len << 20), tmem + kMxSfaCol + 4 * st,
                          tmem + kMxSfbCol + 2 * (n - left));
          else if constexpr (!kDq)
            mma_fp8_k128(issue, d_tmem, a_lo, b_lo, kHi, id_base + (len << 20));
          else
            mma_f16_k128(issue, d_tmem, a_lo, b_lo, kHi, id_base + (len << 20), kQHalfLo);
          left -= len;
          pos += len;
          b_lo += len * kQRowLo;
          // (kChunkCommits) a chunk before the tile's last tells the
          // epilogue that its pairs are in TMEM, so that they are read while
          // the rest of the tile waits for slots
          if (kChunkCommits && left != 0) {
            mma_commit_if(issue, bars.ch(ce));
            ++ce;
          }
        } while (left != 0);
        if (!ok) break;
        // one commit per tile: the K stage is free and every pair of the tile
        // is in TMEM once it fires (each commit costs the issuing thread about
        // as much as a small MMA)
        mma_commit_if(issue, bars.kve(st));
        if constexpr (kDq) mma_commit_if(issue, bars.tr(it, true));
      }
      if (!ok) break;
      mma_commit_if(issue, bars.q_empty);
      ++gi;
    }
    if (leader) {
      // every Q copy has landed before the CTA may exit
      if (nq > 0) wait_drain(bars.q_full, (nq - 1) & 1);
      // No MMA may still be writing TMEM when it is freed.
      mma_commit(bars.mma_done);
      wait_drain(bars.mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kEpiWarps) {
    // =================================================== epilogue
    // Pair p of the CTA's stream (tile's first pair position pos, row r:
    // p = pos + r) sits in TMEM slot p mod kSlots and belongs to warpgroup
    // p mod kEpiWg, so this warp visits r = (wg - pos) mod kEpiWg, + kEpiWg,
    // ... of each tile; the slot's fill index is p / kSlots.
    //   sum_h w_h relu(x_h) = (sum_h w_h x_h + sum_h w_h |x_h|) / 2
    // so the head reduction is 64 packed FMAs (the |x| is an operand
    // modifier) instead of 64 max plus 32 packed FMAs.  The 64 columns come
    // in pieces of kPiece; the slot is released after the last piece is
    // read.
    constexpr int kPiece = 32;
    const uint32_t wg = static_cast<uint32_t>(warp - 4) >> 2;
    const int quarter = warp & 3;    // TMEM lanes this warp may read
    const int tok = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    OutT* const out = static_cast<OutT*>(p.logits);
    uint32_t it = 0, gi = 0, pos = 0, ce = 0;  // tiles, groups, pairs, early chunks seen
    bool ok = true;
    while (ok && walk.next(sched, S, T, p.ctx, walk_ranges, lane)) {
      const int n = walk.n;
      const uint32_t wb = gi & 1;
      ok = warp_wait(bars.wf(wb), (gi >> 1) & 1, abort_flag, p.status);
      if (!ok) break;
      const int lim = static_cast<int>(min(static_cast<int64_t>(walk.npages) * kPageTokens, p.logits_stride));
      const float* w_grp = w_sm + wb * kWBufFloats;
      const int32_t* ctx_grp = ctx_sm + wb * kGroupMaxRows;
      OutT* const out_grp = out + static_cast<int64_t>(walk.r0) * p.logits_stride;
      for (int j = walk.j0; j < walk.j1; ++j, ++it) {
        const uint32_t r_first = (wg - pos) & (kEpiWg - 1);
        // the tile's chunks as the MMA warp forms them (kChunkCommits): pairs
        // [0, e0), [e0, e1), [e1, n); chunks before the last signal on the
        // chunk ring from ce on, the last one with the tile's commit.  A tile
        // of n <= kSlots rows has at most three chunks (one cut where the
        // slot ring wraps, the others at 4 pairs).
        const uint32_t nu = static_cast<uint32_t>(n);
        uint32_t e0 = nu, e1 = nu, nch = 1;
        if constexpr (kChunkCommits) {
          e0 = chunk_len<kSlots>(pos, nu);
          if (e0 < nu) {
            e1 = e0 + chunk_len<kSlots>(pos + e0, nu - e0);
            nch = e1 < nu ? 3 : 2;
          }
        }
        if (r_first >= static_cast<uint32_t>(n)) {  // no pair of this warp in the tile
          pos += static_cast<uint32_t>(n);
          ce += nch - 1;
          continue;
        }
        const int scol = j * kTileTokens + tok;
        const bool in_span = scol < lim;
        float kscale = 1.f;  // (MXFP4: every scale is applied inside the MMA)
        int waited = -1;     // the chunk this warp last waited for
        if constexpr (!kChunkCommits) {
          // the tile's MMAs are done, so its key scales (loaded with its K
          // values, a ring of kScaleStages tiles) are in shared memory too
          ok = warp_wait(bars.tr(it, kDq), (it / kTileRing) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          if (!kMx) kscale = scale_sm[(it & (kScaleStages - 1)) * kScaleStageFloats + tok];
        }
        for (uint32_t r = r_first; r < static_cast<uint32_t>(n); r += kEpiWg) {
          if constexpr (kChunkCommits) {
            const int k = (r >= e0 ? 1 : 0) + (r >= e1 ? 1 : 0);
            if (k != waited) {
              // the chunk's (or the tile's) MMAs are done, and with them the
              // tile's key scales have landed
              if (k + 1 == static_cast<int>(nch))
                ok = warp_wait(bars.tr(it, kDq), (it / kTileRing) & 1, abort_flag, p.status);
              else
                ok = warp_wait(bars.ch(ce + k), ((ce + k) / kChunkRing) & 1, abort_flag, p.status);
              if (!ok) break;
              tc_fence_after();
              if (!kMx && waited < 0) kscale = scale_sm[(it & (kScaleStages - 1)) * kScaleStageFloats + tok];
              waited = k;
            }
          }
          const uint32_t pp = pos + r;
          const uint32_t sl = pp % kSlots;
          const float4* wr = reinterpret_cast<const float4*>(w_grp + r * kHeads);
          float2 cx = make_float2(0.f, 0.f), ca = cx;
#pragma unroll
          for (int pc = 0; pc < kHeads / kPiece; ++pc) {
            uint32_t v[kPiece];
            tmem_ld_cols(t_lane + sl * kPairCols + pc * kPiece, v);
            tmem_ld_wait();
            if (pc == kHeads / kPiece - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bars.te(sl));
            }
#pragma unroll
            for (int h = 0; h < kPiece; h += 4) {
              const float4 w4 = wr[(pc * kPiece + h) / 4];
              const float2 x01 = make_float2(__uint_as_float(v[h + 0]), __uint_as_float(v[h + 1]));
              const float2 x23 = make_float2(__uint_as_float(v[h + 2]), __uint_as_float(v[h + 3]));
              cx = __ffma2_rn(x01, make_float2(w4.x, w4.y), cx);
              ca = __ffma2_rn(make_float2(fabsf(x01.x), fabsf(x01.y)), make_float2(w4.x, w4.y), ca);
              cx = __ffma2_rn(x23, make_float2(w4.z, w4.w), cx);
              ca = __ffma2_rn(make_float2(fabsf(x23.x), fabsf(x23.y)), make_float2(w4.z, w4.w), ca);
            }
          }
          float acc = 0.5f * ((cx.x + cx.y) + (ca.x + ca.y));
          const float logit = (scol < ctx_grp[r]) ? kscale * acc : -INFINITY;
          if (in_span) store_logit(out_grp + static_cast<int64_t>(r) * p.logits_stride + scol, logit);
        }
        if (!ok) break;
        pos += static_cast<uint32_t>(n);
        ce += nch - 1;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.we(wb));
      ++gi;
    }
  }

  // After an abort (a wait that timed out), let any copy still in flight
  // land before the CTA's shared memory and TMEM are given up.
  if (*abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < kDrainTimeoutNs) {
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

namespace {

Params make_params(const LogitsArgs& a) {
  Params p;
  p.q = a.q;
  p.q_scale = a.q_scale;
  p.kv_cache = a.kv_cache;
  p.page_stride = a.page_stride;
  p.num_pages = a.num_pages;
  p.weights = a.weights;
  p.ctx = a.context_lens;
  p.block_table = a.block_table;
  p.bt_stride = a.bt_stride;
  p.bt_rows = a.bt_rows;
  p.bt_num_rows = a.bt_num_rows;
  p.indices = a.indices;
  p.schedule = a.schedule;
  p.num_sms = a.num_sms;
  p.logits = a.logits;
  p.logits_stride = a.logits_stride;
  p.num_rows = a.num_rows;
  p.status = a.status;
  return p;
}

template <int kFmt, typename OutT, bool kChunkCommits>
cudaError_t launch_as(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const Params& p, int grid,
                      cudaStream_t stream) {
  constexpr int kBytes = Smem<kFmt>::kBytes;
  auto* kernel = logits_kernel<kFmt, OutT, kChunkCommits>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBytes);
  if (e != cudaSuccess) return e;
  return launch_dependent(kernel, dim3(grid), dim3(kThreadsOf<kFmt>), kBytes, stream, tm_q, tm_kv, p);
}

// FP8 calls whose rows map onto table rows 8 or more at a time (prefill
// rows reading their request's pages) are walked in full 8-row groups, whose
// tiles fill all 8 TMEM slots: their kernel commits each chunk of a tile's
// MMAs, so that the epilogue reads a tile's first pairs while the rest wait
// for slots.  Decode batches (1-6 rows a group) commit once per tile.
template <int kFmt, typename OutT>
cudaError_t launch_mode(const LogitsArgs& a, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const Params& p,
                          cudaStream_t stream) {
  if constexpr (kFmt == DSA_KV_FP8) {
    if (a.bt_rows != nullptr && a.bt_num_rows > 0 &&
        static_cast<int64_t>(a.num_rows) >= static_cast<int64_t>(kGroupMaxRows) * a.bt_num_rows)
      return launch_as<kFmt, OutT, true>(tm_q, tm_kv, p, a.num_sms, stream);
  }
  return launch_as<kFmt, OutT, false>(tm_q, tm_kv, p, a.num_sms, stream);
}

template <int kFmt>
cudaError_t launch(const LogitsArgs& a, const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const Params& p,
                   cudaStream_t stream) {
  if (a.logits_dtype == DSA_LOGITS_BF16) return launch_mode<kFmt, __nv_bfloat16>(a, tm_q, tm_kv, p, stream);
  return launch_mode<kFmt, float>(a, tm_q, tm_kv, p, stream);
}

}  // namespace

cudaError_t launch_logits_fp8(const LogitsArgs& a, cudaStream_t stream) {
  alignas(64) CUtensorMap tm_q, tm_kv;
  const uint64_t qdims[2] = {static_cast<uint64_t>(kHeadDim),
                             static_cast<uint64_t>(a.num_rows) * kHeads};
  const uint64_t qstrides[1] = {static_cast<uint64_t>(kHeadDim)};
  const uint32_t qbox[2] = {static_cast<uint32_t>(kHeadDim), static_cast<uint32_t>(kHeads)};
  if (!encode_tensor_map_u8(&tm_q, 2, const_cast<uint8_t*>(a.q), qdims, qstrides, qbox, 128))
    return cudaErrorInvalidValue;
  const uint64_t kdims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(kPageTokens),
                             static_cast<uint64_t>(a.num_pages)};
  const uint64_t kstrides[2] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(a.page_stride)};
  const uint32_t kbox[3] = {static_cast<uint32_t>(kHeadDim), static_cast<uint32_t>(kPageTokens), 1};
  if (!encode_tensor_map_u8(&tm_kv, 3, const_cast<uint8_t*>(a.kv_cache), kdims, kstrides, kbox, 128))
    return cudaErrorInvalidValue;
  const Params p = make_params(a);
  return launch<DSA_KV_FP8>(a, tm_q, tm_kv, p, stream);
}

cudaError_t launch_logits_fp4(const LogitsArgs& a, cudaStream_t stream) {
  // The FP4 variant reads its pages with plain bulk copies and converts q
  // itself; the tensor-map parameters are unused.
  alignas(64) CUtensorMap unused{};
  const Params p = make_params(a);
  return launch<DSA_KV_FP4>(a, unused, unused, p, stream);
}

cudaError_t launch_logits_mxfp4(const LogitsArgs& a, cudaStream_t stream) {
  // packed e2m1 q rows and key pages by TMA with the 64-byte swizzle (rows of
  // 64 bytes: 128 elements)
  alignas(64) CUtensorMap tm_q, tm_kv;
  constexpr uint32_t kRowBytes = kHeadDim / 2;
  const uint64_t qdims[2] = {kRowBytes, static_cast<uint64_t>(a.num_rows) * kHeads};
  const uint64_t qstrides[1] = {kRowBytes};
  const uint32_t qbox[2] = {kRowBytes, static_cast<uint32_t>(kHeads)};
  if (!encode_tensor_map_u8(&tm_q, 2, const_cast<uint8_t*>(a.q), qdims, qstrides, qbox, 64))
    return cudaErrorInvalidValue;
  const uint64_t kdims[3] = {kRowBytes, static_cast<uint64_t>(kPageTokens), static_cast<uint64_t>(a.num_pages)};
  const uint64_t kstrides[2] = {kRowBytes, static_cast<uint64_t>(a.page_stride)};
  const uint32_t kbox[3] = {kRowBytes, static_cast<uint32_t>(kPageTokens), 1};
  if (!encode_tensor_map_u8(&tm_kv, 3, const_cast<uint8_t*>(a.kv_cache), kdims, kstrides, kbox, 64))
    return cudaErrorInvalidValue;
  const Params p = make_params(a);
  return launch<DSA_KV_MXFP4>(a, tm_q, tm_kv, p, stream);
}

}  // namespace dsa
