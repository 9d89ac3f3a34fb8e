// tcgen05 tile-attention forward for bf16, head_dim 128, on pairs of SMs
// (cta_group::2, sm_103a).
//
// Computes, for every work item (up to 256 queries and the K/V segments of one
// streaming part: consecutive edges of the task graph, "Context Parallelism
// (CP)" §2.1), the state (O, L): O normalised over the visible keys of the
// part, L = natural-log LSE of the masked scaled scores.  The key tiles stream
// through the online recurrence of "上下文并行" 02 ONE ROW (running max m,
// denominator l, accumulator a in TMEM); the result is a float32 partial state
// for the merge, or, when the part is its Q chunk's only one, the final bf16 O
// and LSE.
//
// A cluster of two CTAs on two SMs runs one item: CTA r holds query rows
// 128 r .. 128 r + 127 and issues nothing to the tensor core; the even CTA
// issues M = 256 MMAs that cover both (cta_group::2):
//   S_b = Q K^T   (M = 256 queries, N = 128 keys, K = 128): each CTA holds its
//                 own Q rows and HALF of the key tile (keys 64 r .. 64 r + 63,
//                 K-major), so one SM reads 6 KB of shared memory per MMA
//                 instead of 8 and loads 16 KB of K per tile instead of 32;
//   O += P_b V    (N = 128 head columns, K = 128 keys): P_b from TMEM, each
//                 CTA holds HALF of the value tile (head columns
//                 64 r .. 64 r + 63, all 128 keys, MN-major).
// TMEM holds two S buffers, two P buffers and O (512 columns).  The softmax
// releases an S buffer as soon as the scores are in its registers and writes
// P into a P buffer of its own, so S of the next key tiles runs on the tensor
// core while the softmax works on this one, and the S MMAs never wait for a
// PV.
// Per CTA, 384 threads (registers: 72 for warps 0..3, 216 for the softmax):
//   warp 0      TMA producer: its Q tile once per item (two buffers), its
//               halves of K and V through 4-stage rings; the bytes of both
//               CTAs are counted on the even CTA's barriers;
//   warp 1      (even CTA) issues S_b = Q K^T for every key tile as soon as
//               the softmax has read S_b of two tiles earlier; TMEM owner in
//               both CTAs;
//   warp 2      (even CTA) issues O += P_b V once both CTAs' P_b is written.
//               Two issuing threads: a thread's first barrier wait after a
//               commit waits for its committed MMAs, and the other thread's
//               queued MMAs keep the tensor core busy meanwhile;
//   warps 4..11 softmax, two warpgroups taking the key tiles in turn (see
//               the softmax section): one query row per thread (its TMEM
//               lane), the 128 scores of a key tile in registers, masks only
//               on tiles that cross the causal or window boundary, exp2 on
//               the MUFU, P written as bf16 pairs into the tile's P buffer, O
//               rescaled in TMEM only when the row max grows by more than 2^8,
//               epilogue O / l and L = (m + log2 l) ln 2.
// Work is a static round-robin of (batch, head, item) over the pairs, items
// sorted heaviest first.  Every main-loop wait is bounded; a CTA that gives up
// raises its own and its peer's abort flag and the device error word, drains
// its copies (and, on the even CTA, its MMAs) and frees TMEM with the peer.
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace cpattn {

namespace {

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;                // per thread at launch (65536 / 384, rounded down to 8)
constexpr int kSmallRegs = 72, kSoftmaxRegs = 216;
static_assert(128 * kSmallRegs + 256 * kSoftmaxRegs == kThreads * kLaunchRegs,
              "register split must add up to the launch total");
constexpr uint32_t kQBytes = 128 * 128 * 2;  // this CTA's Q tile: 32 KB
constexpr uint32_t kQHalf = kQBytes / 2;     // one 64-column box of it
constexpr uint32_t kKBytes = 64 * 128 * 2;   // this CTA's half of a key tile (64 keys): 16 KB
constexpr uint32_t kKHalf = kKBytes / 2;     // one 64-column box of it
constexpr uint32_t kVBytes = 128 * 64 * 2;   // this CTA's half of a value tile (64 columns): 16 KB
constexpr int kQBufs = 2, kKStages = 4, kVStages = 4, kSBufs = 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBufs * kQBytes;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffBar = kOffV + kVStages * kVBytes;
constexpr int kOffX = kOffBar + 512;  // softmax hand-over: running max [2 tile parities][128], and
                                      // per warp its row-sum base and sum [2 warps][2][128]
constexpr int kSmemBytes = kOffX + (2 * 128 + 2 * 2 * 128) * 4;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

// Barrier slots (8 bytes each), the same layout in both CTAs.  "even": only
// the even CTA's copy is used; "both": the MMA commits arrive on both copies.
enum {
  B_QFULL0 = 0,                     // even, + buffer: both CTAs' Q bytes landed
  B_QEMPTY0 = B_QFULL0 + kQBufs,    // both, + buffer: the item's last S has read Q
  B_KFULL0 = B_QEMPTY0 + kQBufs,    // even, + stage
  B_KEMPTY0 = B_KFULL0 + kKStages,  // both, + stage
  B_VFULL0 = B_KEMPTY0 + kKStages,  // even, + stage
  B_VEMPTY0 = B_VFULL0 + kVStages,  // both, + stage
  B_SFULL0 = B_VEMPTY0 + kVStages,  // both, + S buffer: S_b written
  B_SEMPTY0 = B_SFULL0 + kSBufs,    // even, + S buffer: both CTAs have read S_b (8 warp arrivals)
  B_PFULL0 = B_SEMPTY0 + kSBufs,    // even, + P buffer: P written in both CTAs (8 warp arrivals)
  B_PVDONE0 = B_PFULL0 + kSBufs,    // both, + P buffer: the PV that read it is complete
  B_ODONE = B_PVDONE0 + kSBufs,     // both: the item's O is final
  B_OEMPTY,                         // even: both CTAs' epilogues have read O (16 warp arrivals)
  B_DRAIN,                          // both: every MMA of both issuers complete (2 arrivals)
  B_MREADY0,                        // + 2 quarter + parity: the running max after a tile of that parity
  B_COUNT = B_MREADY0 + 8
};
static_assert(8 * B_COUNT + 8 <= 512, "barrier area");

// Opt-in timeline trace (build with -DCPATTN_TRACE): the first pair records
// one clock64 per (event, streamed key tile) for the first kTraceTiles tiles,
// events of the even CTA and of the odd CTA in separate rows (the two SMs'
// clocks are not comparable with each other).
#ifdef CPATTN_TRACE
constexpr int kTraceTiles = 4096, kTraceEvents = 16;
__device__ unsigned long long g_pair_trace[kTraceEvents * kTraceTiles];
#define PAIR_TRACE(ev, tile)                                                       \
  do {                                                                             \
    if (blockIdx.x < 2 && (tile) < unsigned(kTraceTiles))                          \
      g_pair_trace[(ev) * kTraceTiles + (tile)] = clock64();                       \
  } while (0)
#else
#define PAIR_TRACE(ev, tile) do { } while (0)
#endif

constexpr uint32_t kIdescS = tc::idesc_bf16(256, 128, /*b_mn_major=*/0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(256, 128, /*b_mn_major=*/1);
// TMEM columns: S_0, S_1 (128 each, float32 scores), P_0, P_1 (64 each, bf16
// pairs), O (128): 512.  Tile g uses S buffer and P buffer g % 2.
constexpr uint32_t kColP = kSBufs * 128;
constexpr uint32_t kColO = kColP + kSBufs * 64;
static_assert(kColO + 128 == 512, "TMEM columns");
constexpr uint16_t kBothCtas = 0x3;

struct Params {
  CUtensorMap tmq, tmk, tmv;  // Q and V boxes of 64 columns x 128 rows, K boxes of 64 x 64
  FwdArgs a;
  int* err;
  long long wait_limit;  // cycle budget of a main-loop wait in the short-wait copy
  float scale_log2;
  int32_t n_items;
  int64_t total_work;
};

// One item as every role sees it: the streamed key tiles are those that the
// item's last query row can see, segment after segment.
struct Item {
  int32_t row0, pos0, len, out_row0;
  int32_t seg_begin, n_seg;  // key segments: table entries, or the single edge
  int32_t qlast;             // position of the item's last query row
  int32_t n;                 // streamed key tiles
  int32_t rows[2];           // query rows of CTA 0 and CTA 1
};

__device__ __forceinline__ int visible(const Seg& s, int qlast, bool causal) {
  int e = s.len;
  if (causal) e = min(e, qlast - s.pos0 + 1);
  return max(e, 0);
}

__device__ __forceinline__ Seg item_seg(const FwdArgs& a, const Item& it, int s) {
  return a.wide_items ? a.wide_segs[it.seg_begin + s]
                      : Seg{a.edge.kv_row0, a.edge.kv_pos0, a.edge.kv_len, a.edge.win};
}

// Walks an item's streamed key tiles in order, loading each segment once.
struct KeyCursor {
  int s, t0, ntile, eff;
  Seg sg;
  __device__ __forceinline__ void reset() {
    s = -1;
    t0 = ntile = eff = 0;
    sg = Seg{0, 0, 0, 0};
  }
  // Moves forward to the segment holding streamed tile t (t never decreases
  // between resets and t < it.n); returns the tile's key offset in it.
  __device__ __forceinline__ int seek(const FwdArgs& a, const Item& it, int t) {
    while (t >= t0 + ntile && s + 1 < it.n_seg) {
      t0 += ntile;
      ++s;
      sg = item_seg(a, it, s);
      eff = visible(sg, it.qlast, a.causal != 0);
      ntile = (eff + kTile - 1) / kTile;
    }
    return (t - t0) * kTile;
  }
};

__device__ __forceinline__ Item load_item(const FwdArgs& a, int idx) {
  Item it;
  if (a.wide_items) {
    const TileItem t = a.wide_items[idx];
    it.row0 = t.row0;
    it.pos0 = t.pos0;
    it.len = t.len;
    it.out_row0 = t.out_row0;
    it.seg_begin = t.seg_begin;
    it.n_seg = t.seg_count;
  } else {
    it.row0 = a.edge.q_row0 + idx * kWideRows;
    it.pos0 = a.edge.q_pos0 + idx * kWideRows;
    it.len = min(kWideRows, a.edge.q_len - idx * kWideRows);
    it.out_row0 = idx * kWideRows;
    it.seg_begin = 0;
    it.n_seg = 1;
  }
  it.rows[0] = min(it.len, kTile);
  it.rows[1] = it.len - it.rows[0];
  it.qlast = it.pos0 + it.len - 1;
  it.n = 0;
  for (int s = 0; s < it.n_seg; ++s)
    it.n += (visible(item_seg(a, it, s), it.qlast, a.causal != 0) + kTile - 1) / kTile;
  return it;
}

__device__ __forceinline__ void decode_work(const Params& p, int64_t w, int& item, int& b, int& h) {
  const int64_t bh = w / p.n_items;
  item = int(w - bh * p.n_items);
  b = int(bh / p.a.H);
  h = int(bh - int64_t(b) * p.a.H);
}

// Descriptor of K-step kk (16 bf16 along the head dimension) of this CTA's
// 64-key half of a key tile: two 128-byte-swizzled 64-column boxes of 8 KB.
__device__ __forceinline__ uint64_t khalf_step(uint64_t base_desc, int kk) {
  return base_desc + uint64_t((((kk >> 2) * int(kKHalf)) + (kk & 3) * 32) >> 4);
}

// Maximum of the raw scores of a row (keys lo <= j < lo + span when
// kMasked, span >= 0), over four independent chains.
template <bool kMasked>
__device__ __forceinline__ float row_max(const uint32_t* sr, int lo, uint32_t span) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < kTile; j += 2) {
    float s0 = __uint_as_float(sr[j]), s1 = __uint_as_float(sr[j + 1]);
    if (kMasked) {
      s0 = uint32_t(j - lo) < span ? s0 : -INFINITY;
      s1 = uint32_t(j + 1 - lo) < span ? s1 : -INFINITY;
    }
    m4[(j >> 1) & 3] = tc::fmax3(m4[(j >> 1) & 3], s0, s1);
  }
  return tc::fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
}

// P = exp2(s * scale_log2 - mu) over the 128 scores of a row: bf16 pairs are
// written over the row's S columns (keys 2c, 2c+1 -> column c) and the row
// sum of the fp32 values is returned.  kMasked keeps keys lo <= j < lo + span.
template <bool kMasked>
__device__ __forceinline__ float p_pass(const uint32_t* sr, int lo, uint32_t span, float mu, uint64_t sl2x2,
                                        uint32_t tS) {
  const uint64_t nmu = tc::f32x2(-mu, -mu);
  uint64_t ls[4] = {tc::f32x2(0.f, 0.f), tc::f32x2(0.f, 0.f), tc::f32x2(0.f, 0.f), tc::f32x2(0.f, 0.f)};
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int j0 = cc * 32 + 2 * e;
      float x0, x1;
      tc::f32x2_split(tc::ffma2(tc::f32x2(__uint_as_float(sr[j0]), __uint_as_float(sr[j0 + 1])), sl2x2, nmu), x0,
                      x1);
      if (kMasked) {
        x0 = uint32_t(j0 - lo) < span ? x0 : -INFINITY;
        x1 = uint32_t(j0 + 1 - lo) < span ? x1 : -INFINITY;
      }
      const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
      ls[e & 3] = tc::fadd2(ls[e & 3], tc::f32x2(p0, p1));
      pk[e] = tc::pack_bf16x2(p0, p1);
    }
    tc::tmem_st16(tS + cc * 16, pk);
  }
  float x, y;
  tc::f32x2_split(tc::fadd2(tc::fadd2(ls[0], ls[1]), tc::fadd2(ls[2], ls[3])), x, y);
  return x + y;
}

// kShortWaits: the copy launched while cp_debug_set_wait_limit has set a
// short wait budget; the default copy never reads the limit.
template <bool kShortWaits>
__global__ void __launch_bounds__(kThreads, 1) fwd_pair_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  if (sbase & 1023) {  // the swizzled layouts need a 1 KB aligned base (the same in both CTAs)
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 2);
    return;
  }
  const uint32_t rank = tc::cluster_ctarank();  // 0: issues the pair's MMAs
  const bool even = rank == 0;
  const uint32_t sQ = sbase + kOffQ, sK = sbase + kOffK, sV = sbase + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  auto bar = [&](int i) { return tc::smem_u32(bars + i); };
  auto bar_even = [&](int i) { return tc::map_to_rank(bar(i), 0); };  // the even CTA's copy
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * B_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT + 4);
  const uint32_t peer_abort = tc::map_to_rank(tc::smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FwdArgs& a = p.a;

  // A wait that gives up stops the peer too (its abort flag, written remotely).
  auto wt = [&](int b, uint32_t parity) -> bool {
    const bool r = tc::wait_bounded<kShortWaits>(bar(b), parity, abort_flag, p.err, p.wait_limit);
    if (!r) tc::st_remote_u32(peer_abort, 1u);
    return r;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if ((i >= B_PFULL0 && i < B_PFULL0 + kSBufs) || (i >= B_SEMPTY0 && i < B_SEMPTY0 + kSBufs))
        cnt = 8;  // a tile's 4 softmax warps x 2 CTAs
      if (i == B_OEMPTY) cnt = 16;                          // all 8 softmax warps x 2 CTAs
      if (i == B_DRAIN) cnt = 2;                                               // both issuers
      tc::mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // both CTAs' barriers exist before any remote arrival, copy or commit
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int64_t first = tc::cluster_id_x(), stride = tc::n_clusters_x();

  if (warp < 4) {
    tc::setmaxnreg_dec<kSmallRegs>();
  }
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&p.tmq);
      tc::prefetch_tmap(&p.tmk);
      tc::prefetch_tmap(&p.tmv);
      uint32_t qi = 0, kg = 0, vg = 0;
      bool ok = true;
      // loads issued per slot (the even CTA arms the same phases of its barriers)
      uint32_t used_q[kQBufs] = {}, used_k[kKStages] = {}, used_v[kVStages] = {};
      KeyCursor ck, cv;  // K runs one tile ahead of V
      auto load_k = [&](const Item& it, int t, int g_kv, int64_t rbase) -> bool {
        const int kt = ck.seek(a, it, t);
        const int row = int(rbase + ck.sg.row0 + kt) + 64 * int(rank);
        const uint32_t st = kg % kKStages;
        if (!wt(B_KEMPTY0 + st, ((kg / kKStages) & 1) ^ 1)) return false;
        if (even) tc::mbar_arrive_expect_tx(bar(B_KFULL0 + st), 2 * kKBytes);
        const uint32_t fb = bar_even(B_KFULL0 + st);
        tc::tma_load_3d_pair(sK + st * kKBytes, &p.tmk, fb, 0, g_kv, row);
        tc::tma_load_3d_pair(sK + st * kKBytes + kKHalf, &p.tmk, fb, 64, g_kv, row);
        ++used_k[st];
        ++kg;
        return true;
      };
      auto load_v = [&](const Item& it, int t, int g_kv, int64_t rbase) -> bool {
        const int kt = cv.seek(a, it, t);
        const int row = int(rbase + cv.sg.row0 + kt);
        const uint32_t st = vg % kVStages;
        if (!wt(B_VEMPTY0 + st, ((vg / kVStages) & 1) ^ 1)) return false;
        if (even) tc::mbar_arrive_expect_tx(bar(B_VFULL0 + st), 2 * kVBytes);
        tc::tma_load_3d_pair(sV + st * kVBytes, &p.tmv, bar_even(B_VFULL0 + st), 64 * int(rank), g_kv, row);
        ++used_v[st];
        ++vg;
        return true;
      };
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        const int g_kv = h / (a.H / a.Hkv);
        const int64_t rbase = int64_t(b) * a.seqlen;
        const uint32_t qb = qi % kQBufs;
        ok = wt(B_QEMPTY0 + qb, ((qi / kQBufs) & 1) ^ 1);
        if (!ok) break;
        if (even) tc::mbar_arrive_expect_tx(bar(B_QFULL0 + qb), 2 * kQBytes);
        const int row = int(rbase + it.row0) + kTile * int(rank);
        tc::tma_load_3d_pair(sQ + qb * kQBytes, &p.tmq, bar_even(B_QFULL0 + qb), 0, h, row);
        tc::tma_load_3d_pair(sQ + qb * kQBytes + kQHalf, &p.tmq, bar_even(B_QFULL0 + qb), 64, h, row);
        ++used_q[qb];
        ++qi;
        ck.reset();
        cv.reset();
        ok = load_k(it, 0, g_kv, rbase);
        for (int t = 1; t < it.n && ok; ++t) {
          ok = load_k(it, t, g_kv, rbase);
          if (ok) ok = load_v(it, t - 1, g_kv, rbase);
        }
        if (ok) ok = load_v(it, it.n - 1, g_kv, rbase);
      }
      // Drain: every copy this CTA started has landed before the block exits.
      // The even CTA waits for the phases it armed (they count the odd CTA's
      // bytes too); the odd CTA, whose copies complete on the even CTA's
      // barriers, waits until each slot it filled was released (consumed), or
      // for the default budget where the even CTA stopped consuming.
      volatile int never = 0;
      const int first_bar[3] = {even ? B_QFULL0 : B_QEMPTY0, even ? B_KFULL0 : B_KEMPTY0,
                                even ? B_VFULL0 : B_VEMPTY0};
      for (int s = 0; s < kQBufs; ++s)
        if (used_q[s]) tc::mbar_wait(bar(first_bar[0] + s), (used_q[s] - 1) & 1, &never, nullptr);
      for (int s = 0; s < kKStages; ++s)
        if (used_k[s]) tc::mbar_wait(bar(first_bar[1] + s), (used_k[s] - 1) & 1, &never, nullptr);
      for (int s = 0; s < kVStages; ++s)
        if (used_v[s]) tc::mbar_wait(bar(first_bar[2] + s), (used_v[s] - 1) & 1, &never, nullptr);
    }
  } else if (warp == 1) {
    // --------------------------------- S = Q K^T issuer (even CTA only) --
    if (even && lane == 0) {
      uint32_t qi = 0, kg = 0, g = 0;
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        const uint32_t qb = qi % kQBufs;
        ok = wt(B_QFULL0 + qb, (qi / kQBufs) & 1);
        ++qi;
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t qd = tc::kmajor_desc(sQ + qb * kQBytes);
        for (int t = 0; t < it.n && ok; ++t, ++g, ++kg) {
          const uint32_t sb = g % kSBufs;
          // S buffer sb was last read by the softmax of tile g - 2
          if (g >= uint32_t(kSBufs)) {
            ok = wt(B_SEMPTY0 + sb, ((g / kSBufs) - 1) & 1);
            if (!ok) break;
          }
          const uint32_t st = kg % kKStages;
          PAIR_TRACE(0, g);
          ok = wt(B_KFULL0 + st, (kg / kKStages) & 1);
          if (!ok) break;
          PAIR_TRACE(1, g);
          tc::fence_after_sync();
          const uint64_t kd = tc::kmajor_desc(sK + st * kKBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_pair_ss(tmem + sb * 128, tc::kmajor_step(qd, kk), khalf_step(kd, kk), kIdescS, kk > 0 ? 1u : 0u);
          PAIR_TRACE(2, g);
          tc::mma_commit_pair(bar(B_SFULL0 + sb), kBothCtas);
          tc::mma_commit_pair(bar(B_KEMPTY0 + st), kBothCtas);
          if (t == it.n - 1) tc::mma_commit_pair(bar(B_QEMPTY0 + qb), kBothCtas);
        }
      }
      tc::mma_commit_pair(bar(B_DRAIN), kBothCtas);
    }
  } else if (warp == 2) {
    // -------------------------------- O += P V issuer (even CTA only) --
    if (even && lane == 0) {
      uint32_t vg = 0, g = 0, items = 0;
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        // the first PV of an item overwrites O: both epilogues of the previous item have read it
        if (items > 0) {
          ok = wt(B_OEMPTY, (items - 1) & 1);
          if (!ok) break;
        }
        ++items;
        for (int t = 0; t < it.n && ok; ++t, ++g, ++vg) {
          const uint32_t sb = g % kSBufs;
          ok = wt(B_PFULL0 + sb, (g / kSBufs) & 1);
          if (!ok) break;
          PAIR_TRACE(3, g);
          const uint32_t vs = vg % kVStages;
          ok = wt(B_VFULL0 + vs, (vg / kVStages) & 1);
          if (!ok) break;
          PAIR_TRACE(4, g);
          tc::fence_after_sync();
          const uint64_t vd = tc::mnmajor_desc(sV + vs * kVBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // P (bf16 pairs in TMEM) x V (MN-major smem)
            tc::mma_pair_ts(tmem + kColO, tmem + kColP + sb * 64 + kk * 8, tc::mnmajor_step(vd, kk), kIdescPV,
                            (t > 0 || kk > 0) ? 1u : 0u);
          PAIR_TRACE(5, g);
          tc::mma_commit_pair(bar(B_PVDONE0 + sb), kBothCtas);
          tc::mma_commit_pair(bar(B_VEMPTY0 + vs), kBothCtas);
          if (t == it.n - 1) tc::mma_commit_pair(bar(B_ODONE), kBothCtas);
        }
      }
      tc::mma_commit_pair(bar(B_DRAIN), kBothCtas);
    }
  } else if (warp >= 4) {
    tc::setmaxnreg_inc<kSoftmaxRegs>();
    // ----------------------------------------------------- softmax warps --
    // Two warpgroups take the key tiles in turn: warps 4..7 the even tiles of
    // the pair's stream, warps 8..11 the odd ones, so while one warp of an
    // SMSP runs its exponentials the other loads and reduces the next tile.
    // Warp w reads TMEM lanes 32 (w % 4) .. +31: thread `row` of either
    // warpgroup owns query row 128 rank + row.  The running max passes from
    // tile to tile through shared memory (barrier B_MREADY of the lane quarter
    // and the tile's parity): the warp of tile g takes the max after tile g - 1,
    // moves it only when this tile lifts it by more than 2^8, and hands it on.
    // Each warp keeps the row sum of its own tiles against the max of its last
    // tile and rescales it when the max has moved; O (in TMEM) is rescaled by
    // the warp whose tile moved the max, after the previous PV.  At the end of
    // an item the two warps of a quarter combine their sums and each writes 64
    // of the 128 output columns.
    const int half = (warp - 4) >> 2;  // this warp takes the tiles g with g % 2 == half
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO;
    float* mrow = reinterpret_cast<float*>(smem + kOffX);  // [tile parity][row]
    float* xend = mrow + 2 * 128;                           // [warp half][base m, sum][row]
    const uint32_t pair_bar = 1 + quarter;                  // the two warps of this lane quarter
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = tc::f32x2(sl2, sl2);
    uint32_t g = 0, items = 0;
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      int idx, b, h;
      decode_work(p, w, idx, b, h);
      const Item it = load_item(a, idx);
      const int rows_here = it.rows[rank];
      const bool row_ok = row < rows_here;
      const int qpos = it.pos0 + kTile * int(rank) + row;
      float m_own = -INFINITY, l = 0.f;  // this warp's row sum and the max it is taken against
      KeyCursor cur;
      cur.reset();
      for (int t = 0; t < it.n && ok; ++t, ++g) {
        const int kt = cur.seek(a, it, t);
        if (int(g & 1) != half) continue;  // the other warp's tile
        const uint32_t sb = g % kSBufs;
        if (warp == 4 && lane == 0 && rank == 0) PAIR_TRACE(6, g);
        ok = __all_sync(0xffffffffu, wt(B_SFULL0 + sb, (g / kSBufs) & 1));
        if (!ok) break;
        if (warp == 4 && lane == 0) PAIR_TRACE(rank == 0 ? 7 : 13, g);
        tc::fence_after_sync();
        // visible keys of this row in this tile: lo <= j < limit (lo > 0 only
        // under a sliding window: keys more than win - 1 positions back)
        const int kpos0 = cur.sg.pos0 + kt;
        int limit = min(kTile, cur.eff - kt);
        if (a.causal) limit = min(limit, qpos - kpos0 + 1);
        if (!row_ok) limit = 0;
        const int lo = cur.sg.win > 0 ? qpos - cur.sg.win + 1 - kpos0 : 0;
        const bool full = __all_sync(0xffffffffu, limit >= kTile && lo <= 0);
        const uint32_t span = uint32_t(max(limit - max(lo, 0), 0));
        const int lo0 = max(lo, 0);
        const uint32_t tS = tmem + lane_off + sb * 128;
        uint32_t sr[128];
        tc::tmem_ld32(tS, sr);
        tc::tmem_ld32(tS + 32, sr + 32);
        tc::tmem_ld32(tS + 64, sr + 64);
        tc::tmem_ld32(tS + 96, sr + 96);
        tc::tmem_wait_ld();
        // the scores are in registers: S_sb may take the next tile's scores
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(bar_even(B_SEMPTY0 + sb));
        if (warp == 4 && lane == 0 && rank == 0) PAIR_TRACE(8, g);
        const float mx = (full ? row_max<false>(sr, 0, kTile) : row_max<true>(sr, lo0, span)) * sl2;
        // the running max after tile g - 1 (every tile but the stream's first
        // waits, so each barrier is waited once per phase; an item's first tile
        // starts from -inf)
        float m_in = -INFINITY;
        if (g > 0) {
          const uint32_t pq = (g - 1) & 1;
          ok = __all_sync(0xffffffffu, wt(B_MREADY0 + 2 * quarter + int(pq), ((g - 1) >> 1) & 1));
          if (!ok) break;
          if (t > 0) m_in = mrow[pq * 128 + row];
        }
        const float m_up = fmaxf(m_in, mx);
        const bool grow = m_up > m_in + 8.0f;  // also true when m_in is -inf and m_up finite
        const float m = grow ? m_up : m_in;
        mrow[(g & 1) * 128 + row] = m;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(B_MREADY0 + 2 * quarter + int(g & 1)));
        if (warp == 4 && lane == 0 && rank == 0) PAIR_TRACE(9, g);
        if (m != m_own) {  // this warp's sum, against the new max
          l = (m_own == -INFINITY) ? 0.f : l * tc::ex2(m_own - m);
          m_own = m;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        // P buffer sb was last read by the PV of tile g - 2 (this warp waits
        // for every such phase, in order)
        if (g >= uint32_t(kSBufs)) {
          ok = __all_sync(0xffffffffu, wt(B_PVDONE0 + sb, ((g / kSBufs) - 1) & 1));
          if (!ok) break;
          tc::fence_after_sync();
        }
        const uint32_t tP = tmem + lane_off + kColP + sb * 64;
        l += full ? p_pass<false>(sr, 0, kTile, mu, sl2x2, tP) : p_pass<true>(sr, lo0, span, mu, sl2x2, tP);
        if (warp == 4 && lane == 0) PAIR_TRACE(rank == 0 ? 10 : 14, g);
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          // O holds the sum up to tile g - 1 against m_in once the PV that
          // read P of tile g - 1 is complete (the next PV waits for this P).
          // That phase is the latest one of its barrier: PV(g - 3) is
          // complete (PV(g - 2) is, see above) and PV(g + 1) waits for PV(g).
          const float corr = (m_in == -INFINITY) ? 0.f : tc::ex2(m_in - m);
          const uint32_t pb = (g - 1) % kSBufs;
          ok = __all_sync(0xffffffffu, wt(B_PVDONE0 + pb, ((g - 1) / kSBufs) & 1));
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t orr[32];
            tc::tmem_ld32(tO + c * 32, orr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) orr[j] = __float_as_uint(__uint_as_float(orr[j]) * corr);
            tc::tmem_st32(tO + c * 32, orr);
          }
        }
        tc::tmem_wait_st();
        if (warp == 4 && lane == 0 && rank == 0) PAIR_TRACE(11, g);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(bar_even(B_PFULL0 + sb));
        if (warp == 4 && lane == 0) PAIR_TRACE(rank == 0 ? 12 : 15, g);
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue --
      if (it.n > 0) {
        ok = __all_sync(0xffffffffu, wt(B_ODONE, items & 1));
        if (!ok) break;
        tc::fence_after_sync();
      }
      // the row's sum over both warps' tiles against the final max (the
      // larger of the two bases: the max never decreases along the stream)
      xend[half * 256 + row] = m_own;
      xend[half * 256 + 128 + row] = l;
      tc::named_bar(pair_bar, 64);
      const float m_o = xend[(half ^ 1) * 256 + row], l_o = xend[(half ^ 1) * 256 + 128 + row];
      const float m_fin = fmaxf(m_own, m_o);
      float l_all = 0.f;
      if (m_fin != -INFINITY) {
        if (m_own != -INFINITY) l_all += l * tc::ex2(m_own - m_fin);
        if (m_o != -INFINITY) l_all += l_o * tc::ex2(m_o - m_fin);
      }
      tc::named_bar(pair_bar, 64);  // both have read before the next item writes
      // The Q chunk's only part (out_row0 = -1) writes the final O (bf16,
      // round to nearest even) and LSE at its own rows; other parts write a
      // float32 partial state for the merge.  Each warp writes 64 columns.
      const int c0 = 64 * half;
      const bool direct = it.out_row0 < 0;
      const int qrow = kTile * int(rank) + row;
      const int64_t prow_i = direct ? (int64_t(b) * a.seqlen + it.row0 + qrow) * a.H + h
                                    : (int64_t(b) * a.part_rows + it.out_row0 + qrow) * a.H + h;
      const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
      if (rows_here > 0) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t orr[32];
          if (it.n > 0) {
            tc::tmem_ld32(tO + c0 + cc * 32, orr);
            tc::tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) orr[j] = 0u;
          }
          if (row_ok && direct) {
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o_out) + prow_i * 128 + c0) + cc * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t* e = orr + 8 * j;
              dst[j] = make_uint4(tc::pack_bf16x2(__uint_as_float(e[0]) * inv, __uint_as_float(e[1]) * inv),
                                  tc::pack_bf16x2(__uint_as_float(e[2]) * inv, __uint_as_float(e[3]) * inv),
                                  tc::pack_bf16x2(__uint_as_float(e[4]) * inv, __uint_as_float(e[5]) * inv),
                                  tc::pack_bf16x2(__uint_as_float(e[6]) * inv, __uint_as_float(e[7]) * inv));
            }
          } else if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(a.o_part + prow_i * 128 + c0) + cc * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(orr[4 * j]) * inv, __uint_as_float(orr[4 * j + 1]) * inv,
                                   __uint_as_float(orr[4 * j + 2]) * inv, __uint_as_float(orr[4 * j + 3]) * inv);
          }
        }
        if (row_ok && half == 0)
          (direct ? a.lse_out : a.lse_part)[prow_i] =
              l_all > 0.f ? (m_fin + tc::lg2(l_all)) * 0.69314718055994531f : -INFINITY;
      }
      if (it.n > 0) {  // O may be overwritten by the next item's first PV
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_remote(bar_even(B_OEMPTY));
        ++items;
      }
    }
  }

  // Teardown: every MMA of the pair is complete (both CTAs) and both CTAs are
  // done with TMEM before the pair frees it.
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      volatile int never = 0;
      tc::mbar_wait(bar(B_DRAIN), 0, &never, nullptr);
    }
    __syncwarp();
  }
  tc::fence_before_sync();
  tc::cluster_sync();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc_pair(tmem, 512);
}

}  // namespace

#ifdef CPATTN_TRACE
extern "C" int cp_fwd_trace_dump(unsigned long long* out, int max_events) {
  cudaDeviceSynchronize();
  const int n = max_events < kTraceEvents * kTraceTiles ? max_events : kTraceEvents * kTraceTiles;
  cudaMemcpyFromSymbol(out, g_pair_trace, sizeof(unsigned long long) * n);
  return n;
}
#endif

bool tc_available() { return tmap_encoder() != nullptr; }

cp_status launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  const int32_t n_items = a.wide_items ? a.n_wide_items : (a.edge.q_len + kWideRows - 1) / kWideRows;
  if (n_items <= 0) return CP_OK;
  if (a.wide_items && !a.wide_segs) return CP_ERR_INVALID_ARG;
  if (a.dtype != CP_BF16 || a.d != 128) return CP_ERR_UNSUPPORTED;
  const long long limit = wait_limit_cycles();
  const bool short_waits = limit < tc::kWaitCycles;
  auto* kern = short_waits ? fwd_pair_kernel<true> : fwd_pair_kernel<false>;
  // per copy and device: the shared memory limit and the resident pair count,
  // set up by the first launch (under a lock: host threads may race on it)
  static std::atomic<int> max_pairs[2][64] = {};
  static std::mutex setup_mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return CP_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs[short_waits][dev].load(std::memory_order_acquire) == 0) {
    std::lock_guard<std::mutex> lock(setup_mu);
    // The register hand-over inside the kernel assumes the launch count.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return CP_ERR_CUDA;
    if (fa.numRegs != kLaunchRegs) return CP_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return CP_ERR_CUDA;
    // pairs that can be resident at once (a GPC with an odd number of free
    // SMs holds one CTA fewer): the persistent grid is sized to them
    cfg.gridDim = dim3(2 * unsigned(num_sms() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return CP_ERR_UNSUPPORTED;
    max_pairs[short_waits][dev].store(n, std::memory_order_release);
  }
  Params p;
  const int64_t rows = int64_t(a.batch) * a.seqlen;
  if (!make_tmap_rows(&p.tmq, a.q, rows, a.H, 128, 128) ||
      !make_tmap_rows(&p.tmk, a.k, rows, a.Hkv, 128, 64) ||
      !make_tmap_rows(&p.tmv, a.v, rows, a.Hkv, 128, 128))
    return CP_ERR_CUDA;
  p.a = a;
  p.err = device_error_ptr();
  p.wait_limit = limit;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.n_items = n_items;
  p.total_work = int64_t(n_items) * a.batch * a.H;
  const int64_t resident = max_pairs[short_waits][dev].load(std::memory_order_acquire);
  const int64_t pairs = p.total_work < resident ? p.total_work : resident;
  cfg.gridDim = dim3(2 * unsigned(pairs));
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return CP_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
