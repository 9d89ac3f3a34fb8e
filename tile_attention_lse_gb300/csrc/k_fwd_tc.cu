// tcgen05 tile-attention forward for bf16, head_dim 128 (sm_103a).
//
// Computes, for every work item (up to 256 queries and the K/V segments of one
// key owner: one edge of the task graph, "Context Parallelism (CP)" §2.1), the
// partial state A_ij = (O_ij, L_ij): O normalised over the visible keys of the
// item, L = natural-log LSE of the masked scaled scores.  The key tiles stream
// through the online recurrence of "上下文并行" 02 ONE ROW (running max m,
// denominator l, accumulator a in TMEM).
//
// An item holds two 128-row Q tiles that share every streamed K/V tile, so a
// K/V tile fetched from L2 feeds four MMAs instead of two.  Persistent kernel,
// one CTA per SM, 384 threads in three warpgroups:
//   warp 0       TMA producer: Q0 and Q1 once per item; K and V tiles through
//                3- and 2-stage rings (K runs one tile ahead of V), all as
//                128-byte-swizzled boxes of 64 x 128 bf16;
//   warps 1, 2   tcgen05.mma issuers (one lane each), warp 1 for Q tile 0
//                and TMEM owner, warp 2 for Q tile 1: S_i = Q_i K^T
//                (M=N=128, K=16 per instruction, fp32 in TMEM), then
//                O_i += P_i V with P_i read from TMEM over S_i (TS form) and V
//                MN-major from shared memory, then S_i of the next key tile
//                once that PV has read P_i.  The two chains are independent,
//                so the tensor core runs one Q tile's MMAs while the other
//                tile's softmax runs;
//   warp 3       idle (it completes the first warpgroup);
//   warps 4..7   softmax of Q tile 0, warps 8..11 of Q tile 1: one query row
//                per thread (its TMEM lane), all 128 scores of the row in
//                registers, masking by original position only on tiles that
//                cross the causal boundary, exp2 on the MUFU, P written back
//                as bf16 pairs over S, lazy rescale of O (only when the row max
//                grows by more than 2^8), epilogue O / l and
//                L = (m + log2 l) ln 2: a float32 partial state, or, for
//                the only part of a Q chunk, the final bf16 O and LSE.  The two warpgroups' exp phases
//                alternate; the TMEM load and row max of one overlap the
//                other's exponentials.
// TMEM (512 columns): S_0/P_0 0..127, S_1/P_1 128..255, O_0 256..383,
// O_1 384..511.  The first warpgroup hands registers to the softmax
// warpgroups (setmaxnreg: 88 + 2 x 208 per thread = 3 x 168, the launch
// total; the host checks the compiled count before launching).  Work is a static round-robin over (batch, head, item) with
// items sorted heaviest first.  Every mbarrier wait is bounded; on timeout the
// block raises the device error word, drains its copies and MMAs and frees
// TMEM.
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace cpattn {

namespace {

// Opt-in timeline trace (build with -DCPATTN_TRACE): block 0 records one
// clock64 per (event, key tile) for the first kTraceTiles tiles.
#ifdef CPATTN_TRACE
constexpr int kTraceTiles = 4096, kTraceEvents = 16;
__device__ unsigned long long g_fwd_trace[kTraceEvents * kTraceTiles];
// one plain store per (event, tile): no atomics on the traced path
#define FWD_TRACE(ev, tile)                                                        \
  do {                                                                             \
    if (blockIdx.x == 0 && (tile) < unsigned(kTraceTiles))                         \
      g_fwd_trace[(ev) * kTraceTiles + (tile)] = clock64();                        \
  } while (0)
#else
#define FWD_TRACE(ev, tile) do { } while (0)
#endif

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;               // per thread at launch (65536 / 384, rounded down to 8)
constexpr int kProducerRegs = 88, kSoftmaxRegs = 208;
static_assert(128 * kProducerRegs + 256 * kSoftmaxRegs == kThreads * kLaunchRegs,
              "register split must add up to the launch total");
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile = 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 128 x 64 swizzled box
constexpr int kKStages = 3, kVStages = 2;
constexpr int kOffQ = 0;                                  // Q0, Q1
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBar = kOffV + kVStages * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256;
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

// barrier slots (8 bytes each)
enum {
  B_QFULL = 0, B_QEMPTY,
  B_KFULL0, B_KEMPTY0 = B_KFULL0 + kKStages,
  B_VFULL0 = B_KEMPTY0 + kKStages, B_VEMPTY0 = B_VFULL0 + kVStages,
  B_SFULL0 = B_VEMPTY0 + kVStages,  // + i: S_i written
  B_PFULL0 = B_SFULL0 + 2,          // + i: P_i written (128 arrivals)
  B_PVDONE0 = B_PFULL0 + 2,         // + i: PV_i complete (P_i may be overwritten)
  B_ODONE0 = B_PVDONE0 + 2,         // + i: O_i of the item final
  B_DRAIN0 = B_ODONE0 + 2,          // + i: every MMA of issuer i complete
  B_COUNT
};
// after the barriers: abort flag, TMEM base, and the two softmax pacing
// counters (tiles whose P each Q tile's warps have written, four per tile)
static_assert(8 * B_COUNT + 16 <= 256, "barrier area");

constexpr uint32_t kIdescS = tc::idesc_bf16(128, 128, /*b_mn_major=*/0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, /*b_mn_major=*/1);

struct Params {
  CUtensorMap tmq, tmk, tmv;
  FwdArgs a;
  int* err;
  long long wait_limit;  // cycle budget of a main-loop wait (drains use the default)
  float scale_log2;
  int32_t n_items;
  int64_t total_work;
};

// One item as every role sees it.  The streamed key tiles are those that the
// item's last query row can see, segment after segment; Q tile i processes
// the first n_q[i] of them (the tiles that tile 0 sees form a prefix of the
// stream because the segments are disjoint and ordered by position; where
// they are not, tile 0 takes the whole stream and masking does the rest).
struct Item {
  int32_t row0, pos0, len, out_row0;
  int32_t seg_begin, n_seg;  // key segments: table entries, or the single edge
  int32_t qlast;             // position of the item's last query row
  int32_t n;                 // streamed key tiles
  int32_t rows[2];           // query rows of Q tile 0 and 1
  int32_t n_q[2];            // key tiles that Q tile 0 and 1 process
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
  const bool causal = a.causal != 0;
  it.qlast = it.pos0 + it.len - 1;
  const int qlast0 = it.pos0 + it.rows[0] - 1;
  // tile 0's visible tiles are a prefix of the stream unless a segment after
  // one that tile 0 sees only in part is visible to tile 0 again
  int n0 = 0;
  bool cut = false, prefix = true;
  it.n = 0;
  for (int s = 0; s < it.n_seg; ++s) {
    const Seg sg = item_seg(a, it, s);
    const int nt = (visible(sg, it.qlast, causal) + kTile - 1) / kTile;
    const int nt0 = (visible(sg, qlast0, causal) + kTile - 1) / kTile;
    if (cut && nt0 > 0) prefix = false;
    if (nt0 < nt) cut = true;
    it.n += nt;
    n0 += nt0;
  }
  it.n_q[0] = prefix ? n0 : it.n;
  it.n_q[1] = it.rows[1] > 0 ? it.n : 0;
  return it;
}

__device__ __forceinline__ void decode_work(const Params& p, int64_t w, int& item, int& b, int& h) {
  const int64_t bh = w / p.n_items;
  item = int(w - bh * p.n_items);
  b = int(bh / p.a.H);
  h = int(bh - int64_t(b) * p.a.H);
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
  float a, b;
  tc::f32x2_split(tc::fadd2(tc::fadd2(ls[0], ls[1]), tc::fadd2(ls[2], ls[3])), a, b);
  return a + b;
}

// kShortWaits: the instantiation launched while cp_debug_set_wait_limit has
// set a short wait budget (main-loop waits probe without suspending and give
// up after Params::wait_limit cycles); the default one never reads the limit.
template <bool kShortWaits>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  if (sbase & 1023) {  // the swizzled layouts need a 1 KB aligned base
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 2);
    return;
  }
  const uint32_t sQ = sbase + kOffQ, sK = sbase + kOffK, sV = sbase + kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  auto bar = [&](int i) { return tc::smem_u32(bars + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * B_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT + 4);
  uint32_t* pace = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT + 8);  // [2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FwdArgs& a = p.a;

  if (threadIdx.x == 0) {
    // operand slots are released by both issuers
    tc::mbar_init(bar(B_QFULL), 1);
    tc::mbar_init(bar(B_QEMPTY), 2);
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(bar(B_KFULL0 + s), 1);
      tc::mbar_init(bar(B_KEMPTY0 + s), 2);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(bar(B_VFULL0 + s), 1);
      tc::mbar_init(bar(B_VEMPTY0 + s), 2);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(B_SFULL0 + i), 1);
      tc::mbar_init(bar(B_PFULL0 + i), 128);  // the four warps of Q tile i
      tc::mbar_init(bar(B_PVDONE0 + i), 1);
      tc::mbar_init(bar(B_ODONE0 + i), 1);
      tc::mbar_init(bar(B_DRAIN0 + i), 1);
    }
    pace[0] = pace[1] = 0;
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int64_t first = blockIdx.x, stride = gridDim.x;

  if (warp < 4) {
    tc::setmaxnreg_dec<kProducerRegs>();
  }
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&p.tmq);
      tc::prefetch_tmap(&p.tmk);
      tc::prefetch_tmap(&p.tmv);
      uint32_t kg = 0, vg = 0, qi = 0;
      bool ok = true;
      uint32_t armed_q = 0, armed_k[kKStages] = {}, armed_v[kVStages] = {};  // uses armed so far
      KeyCursor ck, cv;  // K runs one tile ahead of V
      auto load_k = [&](const Item& it, int t, int g_kv, int64_t rbase) -> bool {
        const int kt = ck.seek(a, it, t);
        const int row = int(rbase + ck.sg.row0 + kt);
        const uint32_t st = kg % kKStages;
        if (!tc::wait_bounded<kShortWaits>(bar(B_KEMPTY0 + st), ((kg / kKStages) & 1) ^ 1, abort_flag, p.err, p.wait_limit)) return false;
        tc::mbar_arrive_expect_tx(bar(B_KFULL0 + st), kTileBytes);
        tc::tma_load_3d(sK + st * kTileBytes, &p.tmk, bar(B_KFULL0 + st), 0, g_kv, row);
        tc::tma_load_3d(sK + st * kTileBytes + kHalfBytes, &p.tmk, bar(B_KFULL0 + st), 64, g_kv, row);
        ++armed_k[st];
        FWD_TRACE(0, kg);
        ++kg;
        return true;
      };
      auto load_v = [&](const Item& it, int t, int g_kv, int64_t rbase) -> bool {
        const int kt = cv.seek(a, it, t);
        const int row = int(rbase + cv.sg.row0 + kt);
        const uint32_t st = vg % kVStages;
        if (!tc::wait_bounded<kShortWaits>(bar(B_VEMPTY0 + st), ((vg / kVStages) & 1) ^ 1, abort_flag, p.err, p.wait_limit)) return false;
        tc::mbar_arrive_expect_tx(bar(B_VFULL0 + st), kTileBytes);
        tc::tma_load_3d(sV + st * kTileBytes, &p.tmv, bar(B_VFULL0 + st), 0, g_kv, row);
        tc::tma_load_3d(sV + st * kTileBytes + kHalfBytes, &p.tmv, bar(B_VFULL0 + st), 64, g_kv, row);
        ++armed_v[st];
        FWD_TRACE(1, vg);
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
        // Q tiles (the second only when it has rows)
        ok = tc::wait_bounded<kShortWaits>(bar(B_QEMPTY), (qi & 1) ^ 1, abort_flag, p.err, p.wait_limit);
        if (!ok) break;
        const bool two = it.rows[1] > 0;
        tc::mbar_arrive_expect_tx(bar(B_QFULL), two ? 2 * kTileBytes : kTileBytes);
        for (int i = 0; i < (two ? 2 : 1); ++i) {
          const int row = int(rbase + it.row0 + i * kTile);
          tc::tma_load_3d(sQ + i * kTileBytes, &p.tmq, bar(B_QFULL), 0, h, row);
          tc::tma_load_3d(sQ + i * kTileBytes + kHalfBytes, &p.tmq, bar(B_QFULL), 64, h, row);
        }
        ++armed_q;
        ++qi;
        // K one tile ahead of V inside the item
        ck.reset();
        cv.reset();
        ok = load_k(it, 0, g_kv, rbase);
        for (int t = 1; t < it.n && ok; ++t) {
          ok = load_k(it, t, g_kv, rbase);
          if (ok) ok = load_v(it, t - 1, g_kv, rbase);
        }
        if (ok) ok = load_v(it, it.n - 1, g_kv, rbase);
      }
      // Drain: every copy this thread started has landed before the block exits.
      volatile int never = 0;
      if (armed_q) tc::mbar_wait(bar(B_QFULL), (armed_q - 1) & 1, &never, nullptr);
      for (int s = 0; s < kKStages; ++s)
        if (armed_k[s]) tc::mbar_wait(bar(B_KFULL0 + s), (armed_k[s] - 1) & 1, &never, nullptr);
      for (int s = 0; s < kVStages; ++s)
        if (armed_v[s]) tc::mbar_wait(bar(B_VFULL0 + s), (armed_v[s] - 1) & 1, &never, nullptr);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------- MMA issuers, one per Q tile --
    if (lane == 0) {
      const int i = warp - 1;
      const uint64_t qd = tc::kmajor_desc(sQ + i * kTileBytes);
      const uint32_t scol = tmem + i * 128, ocol = tmem + 256 + i * 128;
      uint32_t kg = 0, vg = 0, qi = 0, pc = 0, pvc = 0;
      bool pv_pending = false;  // a PV_i whose completion S_i has not waited for
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        const int nq = it.n_q[i];
        ok = tc::wait_bounded<kShortWaits>(bar(B_QFULL), qi & 1, abort_flag, p.err, p.wait_limit);
        ++qi;
        if (!ok) break;
        tc::fence_after_sync();
        if (nq == 0) tc::mbar_arrive(bar(B_QEMPTY));  // this tile reads no Q here
        for (int t = 0; t < it.n && ok; ++t) {
          // S_i = Q_i K^T, after PV_i of the previous key tile has read P_i
          const uint32_t st = kg % kKStages;
          ok = tc::wait_bounded<kShortWaits>(bar(B_KFULL0 + st), (kg / kKStages) & 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          if (i == 1) FWD_TRACE(6, kg);
          if (t < nq) {
            if (pv_pending) {
              ok = tc::wait_bounded<kShortWaits>(bar(B_PVDONE0 + i), (pvc - 1) & 1, abort_flag, p.err, p.wait_limit);
              if (!ok) break;
              pv_pending = false;
            }
            tc::fence_after_sync();
            const uint64_t kd = tc::kmajor_desc(sK + st * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc::mma_ss(scol, tc::kmajor_step(qd, kk), tc::kmajor_step(kd, kk), kIdescS, kk > 0 ? 1u : 0u);
            tc::mma_commit(bar(B_SFULL0 + i));
            tc::mma_commit(bar(B_KEMPTY0 + st));
            if (t == nq - 1) tc::mma_commit(bar(B_QEMPTY));
            FWD_TRACE(2 + 6 * i, kg);
          } else {
            tc::mbar_arrive(bar(B_KEMPTY0 + st));  // this tile does not read K here
          }
          ++kg;
          // O_i += P_i V
          const uint32_t vs = vg % kVStages;
          ok = tc::wait_bounded<kShortWaits>(bar(B_VFULL0 + vs), (vg / kVStages) & 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          if (t < nq) {
            ok = tc::wait_bounded<kShortWaits>(bar(B_PFULL0 + i), pc & 1, abort_flag, p.err, p.wait_limit);
            ++pc;
            if (!ok) break;
            FWD_TRACE(4 + i, vg);
            tc::fence_after_sync();
            const uint64_t vd = tc::mnmajor_desc(sV + vs * kTileBytes);
            const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // P (bf16 pairs in TMEM) x V (MN-major smem)
              tc::mma_ts(ocol, scol + kk * 8, tc::mnmajor_step(vd, kk), kIdescPV, kk == 0 ? acc0 : 1u);
            tc::mma_commit(bar(B_PVDONE0 + i));
            pv_pending = true;
            ++pvc;
            tc::mma_commit(bar(B_VEMPTY0 + vs));
            if (t == nq - 1) tc::mma_commit(bar(B_ODONE0 + i));  // O_i of this item is final
            FWD_TRACE(3 + 4 * i, vg);
          } else {
            tc::mbar_arrive(bar(B_VEMPTY0 + vs));
          }
          ++vg;
        }
      }
      // Drain: all MMAs issued by this thread are complete before TMEM is freed.
      volatile int never = 0;
      tc::mma_commit(bar(B_DRAIN0 + i));
      tc::mbar_wait(bar(B_DRAIN0 + i), 0, &never, nullptr);
    }
#ifdef CPATTN_TRACE
  } else if (warp == 3) {
    // trace only: when each K and V tile lands
    if (lane == 0) {
      uint32_t kg = 0, vg = 0;
      volatile int never = 0;
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        for (int t = 0; t < it.n && ok; ++t) {
          ok = tc::mbar_wait(bar(B_KFULL0 + kg % kKStages), (kg / kKStages) & 1, abort_flag, nullptr);
          ++kg;
          if (ok) ok = tc::mbar_wait(bar(B_VFULL0 + vg % kVStages), (vg / kVStages) & 1, abort_flag, nullptr);
          ++vg;
        }
      }
      (void)never;
    }
#endif
  } else if (warp >= 4) {
    tc::setmaxnreg_inc<kSoftmaxRegs>();
    // ----------------------------------------------------- softmax warps --
    // Warps 4..7 serve Q tile 0, warps 8..11 Q tile 1; warp w reads TMEM lanes
    // 32 (w % 4) .. +31, so thread `row` owns query row `row` of its tile.
    const int qt = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + qt * 128, tO = tmem + lane_off + 256 + qt * 128;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = tc::f32x2(sl2, sl2);
    uint32_t sc = 0, oc = 0;
    uint32_t pbase = 0;  // key tiles of the other Q tile in earlier items
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      int idx, b, h;
      decode_work(p, w, idx, b, h);
      const Item it = load_item(a, idx);
      const int nq = it.n_q[qt];
      const int qpos = it.pos0 + qt * kTile + row;
      float m = -INFINITY, l = 0.f;
      KeyCursor cur;
      cur.reset();
      for (int t = 0; t < nq && ok; ++t) {
        const int kt = cur.seek(a, it, t);
        ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_SFULL0 + qt), sc & 1, abort_flag, p.err, p.wait_limit));
        ++sc;
        if (!ok) break;
        tc::fence_after_sync();
        if (lane == 0 && quarter == 0) FWD_TRACE(13 + qt, sc - 1);
        // visible keys of this row in this tile: lo <= j < limit (lo > 0 only
        // under a sliding window: keys more than win - 1 positions back)
        const int kpos0 = cur.sg.pos0 + kt;
        int limit = min(kTile, cur.eff - kt);
        if (a.causal) limit = min(limit, qpos - kpos0 + 1);
        const int lo = cur.sg.win > 0 ? qpos - cur.sg.win + 1 - kpos0 : 0;
        const bool full = __all_sync(0xffffffffu, limit >= kTile && lo <= 0);
        const uint32_t span = uint32_t(max(limit - max(lo, 0), 0));
        const int lo0 = max(lo, 0);
        uint32_t sr[128];
        tc::tmem_ld32(tS, sr);
        tc::tmem_ld32(tS + 32, sr + 32);
        tc::tmem_ld32(tS + 64, sr + 64);
        tc::tmem_ld32(tS + 96, sr + 96);
        tc::tmem_wait_ld();
        // row max and the running-max update run while the other Q tile's
        // warps are in their exp phase
        const float mx = (full ? row_max<false>(sr, 0, kTile) : row_max<true>(sr, lo0, span)) * sl2;
        const float m_new = fmaxf(m, mx);
        const bool grow = m_new > m + 8.0f;  // also true when m is -inf and m_new finite
        float corr = 1.f;
        if (grow) {
          corr = (m == -INFINITY) ? 0.f : tc::ex2(m - m_new);
          m = m_new;
          l *= corr;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        // The exp phases of the two Q tiles alternate (they share the SFU and
        // convert pipe): tile 1 starts after tile 0 has written P for the
        // same key tile, tile 0 after tile 1 has written P for the previous
        // key tile.  The counters only pace the warps; no data flows through
        // them.
        if (qt == 1) {
          if (t < it.n_q[0])
            ok = __all_sync(0xffffffffu, tc::wait_count<kShortWaits>(pace + 0, 4 * (pbase + t + 1), abort_flag, p.err, p.wait_limit));
        } else if (t > 0 && t - 1 < it.n_q[1]) {
          ok = __all_sync(0xffffffffu, tc::wait_count<kShortWaits>(pace + 1, 4 * (pbase + t), abort_flag, p.err, p.wait_limit));
        }
        if (!ok) break;
        if (lane == 0 && quarter == 0) FWD_TRACE(11 + qt, sc - 1);
        const float lsum =
            full ? p_pass<false>(sr, 0, kTile, mu, sl2x2, tS) : p_pass<true>(sr, lo0, span, mu, sl2x2, tS);
        l += lsum;
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          // S_i of this tile was issued after PV_i of the previous one
          // completed, so O_i is final up to the previous tile here (and PV_i
          // of this tile waits for the P-full arrival below).
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
        tc::fence_before_sync();
        tc::mbar_arrive(bar(B_PFULL0 + qt));
        if (lane == 0) atomicAdd(pace + qt, 1u);
        if (lane == 0 && quarter == 0) FWD_TRACE(9 + qt, sc - 1);
      }
      pbase += it.n_q[qt ^ 1];
      if (!ok) break;
      // ------------------------------------------------------ epilogue --
      if (it.rows[qt] == 0) continue;  // no query rows in this tile (no MMAs either)
      if (nq > 0) {
        ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_ODONE0 + qt), oc & 1, abort_flag, p.err, p.wait_limit));
        ++oc;
        if (!ok) break;
        tc::fence_after_sync();
      }
      const bool store = row < it.rows[qt];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // The Q chunk's only part (out_row0 = -1) writes the final O (bf16,
      // round to nearest even) and LSE at its own rows; other parts write a
      // float32 partial state for the merge.
      const bool direct = it.out_row0 < 0;
      const int qrow = qt * kTile + row;
      const int64_t prow_i = direct ? (int64_t(b) * a.seqlen + it.row0 + qrow) * a.H + h
                                    : (int64_t(b) * a.part_rows + it.out_row0 + qrow) * a.H + h;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t orr[32];
        if (nq > 0) {
          tc::tmem_ld32(tO + cc * 32, orr);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) orr[j] = 0u;
        }
        if (store && direct) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o_out) + prow_i * 128) + cc * 4;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t* e = orr + 8 * j;
            dst[j] = make_uint4(tc::pack_bf16x2(__uint_as_float(e[0]) * inv, __uint_as_float(e[1]) * inv),
                                tc::pack_bf16x2(__uint_as_float(e[2]) * inv, __uint_as_float(e[3]) * inv),
                                tc::pack_bf16x2(__uint_as_float(e[4]) * inv, __uint_as_float(e[5]) * inv),
                                tc::pack_bf16x2(__uint_as_float(e[6]) * inv, __uint_as_float(e[7]) * inv));
          }
        } else if (store) {
          float4* dst = reinterpret_cast<float4*>(a.o_part + prow_i * 128) + cc * 8;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(orr[4 * j]) * inv, __uint_as_float(orr[4 * j + 1]) * inv,
                                 __uint_as_float(orr[4 * j + 2]) * inv, __uint_as_float(orr[4 * j + 3]) * inv);
        }
      }
      tc::fence_before_sync();
      if (store) (direct ? a.lse_out : a.lse_part)[prow_i] = l > 0.f ? (m + tc::lg2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool tc_available() { return tmap_encoder() != nullptr; }

#ifdef CPATTN_TRACE
extern "C" int cp_fwd_trace_dump(unsigned long long* out, int max_events) {
  cudaDeviceSynchronize();
  const int n = max_events < kTraceEvents * kTraceTiles ? max_events : kTraceEvents * kTraceTiles;
  cudaMemcpyFromSymbol(out, g_fwd_trace, sizeof(unsigned long long) * n);
  return n;
}
#endif

cp_status launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  const int32_t n_items = a.wide_items ? a.n_wide_items : (a.edge.q_len + kWideRows - 1) / kWideRows;
  if (n_items <= 0) return CP_OK;
  if (a.wide_items && !a.wide_segs) return CP_ERR_INVALID_ARG;
  if (a.dtype != CP_BF16 || a.d != 128) return CP_ERR_UNSUPPORTED;
  const long long limit = wait_limit_cycles();
  const bool short_waits = limit < tc::kWaitCycles;
  auto* kern = short_waits ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[short_waits][dev]) {
    // The register hand-over inside the kernel assumes the launch count.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return CP_ERR_CUDA;
    if (fa.numRegs != kLaunchRegs) return CP_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return CP_ERR_CUDA;
    attr_set[short_waits][dev] = true;
  }
  Params p;
  const int64_t rows = int64_t(a.batch) * a.seqlen;
  if (!make_tmap_rows(&p.tmq, a.q, rows, a.H, 128, 128) ||
      !make_tmap_rows(&p.tmk, a.k, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmv, a.v, rows, a.Hkv, 128, 128))
    return CP_ERR_CUDA;
  p.a = a;
  p.err = device_error_ptr();
  p.wait_limit = limit;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.n_items = n_items;
  p.total_work = int64_t(n_items) * a.batch * a.H;
  const int64_t grid = p.total_work < num_sms() ? p.total_work : num_sms();
  kern<<<unsigned(grid), kThreads, kSmemBytes, s>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
