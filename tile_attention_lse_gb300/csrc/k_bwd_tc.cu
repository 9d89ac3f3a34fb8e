// tcgen05 tile-attention backward for bf16, head_dim 128 (sm_103a).
//
// "上下文并行" 01 BACKWARD/REPLAY and GRADIENT/RETURN: every block of the
// task graph is replayed from the merged row LSE (P = exp(S - L)) and
// D = <dO, O>; with dS = P (dP - D)
//   dV_j += sum_i P_ij dO_i,   dK_j += scale sum_i dS_ij Q_i,   dQ_i += scale sum_j dS_ij K_j.
// One persistent kernel plus a conversion pass:
//
// dkdv_kernel — one item = one K/V tile (128 keys, one kv-head) plus every Q
//   range of every query rank that sees it (ring order) and every q-head of
//   the group, so the dK/dV contributions of all query ranks are summed in
//   TMEM at the key owner and written once.  Per query tile:
//     S^T  = K Q^T   -> TMEM [0,128)    P^T (bf16) is written over it
//     dP^T = V dO^T  -> TMEM [128,256)
//     dV  += P^T dO  (A = P^T from TMEM, dO read MN-major) -> TMEM [256,384)
//     dK  += dS^T Q  (A = dS^T from shared memory, Q MN-major) -> TMEM [384,512)
//     dQ_t = dS K    (A = the same dS^T tile read MN-major, K MN-major)
//                    -> TMEM [128,256) once dS^T has been taken from dP^T
//   Issue order dP(i), dV(i), S(i+1), dQ(i), dK(i), dP(i+1), ... : dP(i)
//   (which needs no P) runs while the math warps build P^T(i), so dP^T is
//   ready when they turn to dS^T; the key-row math of tile i+1 (P^T)
//   overlaps dQ(i) and dK(i); dQ(i) goes first so that its read-out, which
//   frees the columns dP(i+1) writes, overlaps dK(i).  Four dQ warps read dQ(i) out of TMEM, hand
//   the columns back for dP(i+1), stage it in shared memory in 32-column
//   chunks and add each chunk into a float32 accumulator with a TMA
//   reduction (the query owner's sum over key owners, resolved in L2;
//   summation order is not fixed).  The reductions leave the SM only at the
//   rate L2 accepts them; issued as per-thread vector reductions they back up
//   the SM's load/store queue and every shared-memory load waits behind them,
//   while the TMA path leaves that queue alone.
//   Warps: 0 TMA, 1 MMA (+TMEM owner), 2 stages L*log2e and D of the query
//   tile, 3 idle, 4..11 key-row math (two warps per TMEM lane quarter, each
//   on 64 query columns: P^T, dS^T, masks, the epilogue), 12..15 dQ read-out
//   and reductions (one per lane quarter).  Registers move between the
//   warpgroups with setmaxnreg.
//
// dq_post_kernel — dQ = scale * accumulator, converted to bf16 [b][s][h][d].
//
// The accumulator is float32 [batch * q-heads][seqlen][128].  Rows of a
// query tile past its end hold exact zeros (their P is 0), so a chunk may be
// reduced over all 128 rows; rows past seqlen are clipped by the tensor map.
//
// P^T written over S^T keeps each warp's half in its own 64 columns (bf16
// pairs in the first 32 of them); the dV MMA reads K-step kk from column
// 64 (kk / 4) + 8 (kk % 4).
//
// Every mbarrier is waited once per phase, in order, so a parity wait can
// never be two phases behind; every wait is bounded (device error word and
// orderly exit).
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace cpattn {

namespace {

constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kHalfBytes = kTileBytes / 2;

constexpr uint32_t kIdescKK = tc::idesc_bf16(128, 128, 0, 0);  // A, B K-major
constexpr uint32_t kIdescKM = tc::idesc_bf16(128, 128, 1, 0);  // B MN-major
constexpr uint32_t kIdescMM = tc::idesc_bf16(128, 128, 1, 1);  // A and B MN-major

struct Params {
  CUtensorMap tmq, tmk, tmv, tmdo, tmdq;
  BwdArgs a;
  int* err;
  long long wait_limit;  // cycle budget of a main-loop wait (drains use the default)
  float scale_log2;
};

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t* r, float mul) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint4 v;
    v.x = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * mul, __uint_as_float(r[8 * q4 + 1]) * mul);
    v.y = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * mul, __uint_as_float(r[8 * q4 + 3]) * mul);
    v.z = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * mul, __uint_as_float(r[8 * q4 + 5]) * mul);
    v.w = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * mul, __uint_as_float(r[8 * q4 + 7]) * mul);
    *reinterpret_cast<uint4*>(dst + q4 * 8) = v;
  }
}

// A value the compiler has to take as computed here: the MMA issuer makes each
// group's base descriptors opaque, so every step costs one add instead of the
// whole unrolled set of 64-bit descriptors staying live across the loop.
__device__ __forceinline__ uint64_t opaque(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// =========================================================== dK / dV ======
namespace kv {

// Opt-in timeline trace (build with -DCPATTN_TRACE): block 0 records one
// clock64 per (event, query tile) for the first kTraceTiles tiles.
#ifdef CPATTN_TRACE
constexpr int kTraceTiles = 4096, kTraceEvents = 16;
__device__ unsigned long long g_kv_trace[kTraceEvents * kTraceTiles];
#define KV_TRACE(ev, tile)                                                          \
  do {                                                                             \
    if (blockIdx.x == 0 && (tile) < unsigned(kTraceTiles))                         \
      g_kv_trace[(ev) * kTraceTiles + (tile)] = clock64();                         \
  } while (0)
#else
#define KV_TRACE(ev, tile) do { } while (0)
#endif

constexpr int kThreads = 512;
constexpr int kLaunchRegs = 128;  // per thread at launch (65536 / 512)
constexpr int kSmallRegs = 72;    // warpgroup 0: TMA, MMA, L/D staging
constexpr int kMathRegs = 144;    // warpgroups 1, 2: key-row math
constexpr int kDqRegs = 152;      // warpgroup 3: dQ read-out (128 columns per thread)
static_assert(128 * (kSmallRegs + kDqRegs) + 256 * kMathRegs == kThreads * kLaunchRegs,
              "setmaxnreg shares must add up to the launch allocation");
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;        // 2 stages
constexpr int kOffDO = kOffQ + 2 * kTileBytes;   // 1 stage
constexpr int kDqChunkBytes = 128 * 32 * 4;       // float32, 32 columns x 128 rows
constexpr int kOffDQ = kOffDO + kTileBytes;      // 2 dQ staging chunks
constexpr int kOffDS = kOffDQ + 2 * kDqChunkBytes;
constexpr int kOffL = kOffDS + kTileBytes;       // 2 stages x 128 floats
constexpr int kOffD = kOffL + 2 * 512;
constexpr int kOffBar = kOffD + 2 * 512;
constexpr int kSmemBytes = kOffBar + 256;

enum {
  B_KVFULL = 0, B_KVEMPTY, B_QFULL0, B_QFULL1, B_QEMPTY0, B_QEMPTY1, B_DOFULL, B_DOEMPTY, B_SFULL, B_DPFULL, B_PFULL, B_PCONS, B_DSFULL, B_DKDV,
  B_LDFULL0, B_LDFULL1, B_LDEMPTY0, B_LDEMPTY1, B_DQFULL, B_DQCONS, B_DRAIN, B_COUNT
};
static_assert(8 * B_COUNT + 8 <= 256, "barrier area");

struct Item {
  int32_t row0, pos0, len, seg_begin, seg_count;
  int b, g, n_tiles;
};

__device__ __forceinline__ Item load_item(const Params& p, int64_t w) {
  const BwdArgs& a = p.a;
  const int64_t bh = w / a.n_kv_items;
  const TileItem t = a.kv_items[int(w - bh * a.n_kv_items)];
  Item it;
  it.b = int(bh / a.Hkv);
  it.g = int(bh - int64_t(it.b) * a.Hkv);
  it.row0 = t.row0;
  it.pos0 = t.pos0;
  it.len = t.len;
  it.seg_begin = t.seg_begin;
  it.seg_count = t.seg_count;
  int n = 0;
  for (int s = 0; s < t.seg_count; ++s) n += (max(a.kv_segs[t.seg_begin + s].len, 0) + kTile - 1) / kTile;
  it.n_tiles = n * (a.H / a.Hkv);
  return it;
}

// Query tiles of an item, in order: q-head of the group, segment, 128 rows.
struct Walk {
  int hj, si, u;
};
struct QTile {
  int h, q0, qpos0, qlen, win;
};

__device__ __forceinline__ void walk_skip_empty(const BwdArgs& a, const Item& it, Walk& w) {
  const int group = a.H / a.Hkv;
  while (w.hj < group && a.kv_segs[it.seg_begin + w.si].len <= 0) {
    if (++w.si == it.seg_count) {
      w.si = 0;
      ++w.hj;
    }
  }
}

__device__ __forceinline__ Walk walk_begin(const BwdArgs& a, const Item& it) {
  Walk w{0, 0, 0};
  walk_skip_empty(a, it, w);
  return w;
}

__device__ __forceinline__ void walk_next(const BwdArgs& a, const Item& it, Walk& w) {
  if ((w.u + 1) * kTile < a.kv_segs[it.seg_begin + w.si].len) {
    ++w.u;
    return;
  }
  w.u = 0;
  if (++w.si == it.seg_count) {
    w.si = 0;
    ++w.hj;
  }
  walk_skip_empty(a, it, w);
}

__device__ __forceinline__ QTile walk_tile(const BwdArgs& a, const Item& it, const Walk& w) {
  const Seg sg = a.kv_segs[it.seg_begin + w.si];
  QTile t;
  t.h = it.g * (a.H / a.Hkv) + w.hj;
  t.q0 = sg.row0 + w.u * kTile;
  t.qpos0 = sg.pos0 + w.u * kTile;
  t.qlen = min(kTile, sg.len - w.u * kTile);
  t.win = sg.win;
  return t;
}

// kShortWaits: the instantiation launched while cp_debug_set_wait_limit has
// set a short wait budget; the default one never reads the limit.
template <bool kShortWaits>
__global__ void __launch_bounds__(kThreads, 1) dkdv_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  if (sbase & 1023) {  // swizzled operand layouts need a 1 KB aligned base
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 2);
    return;
  }
  const uint32_t sK = sbase + kOffK, sV = sbase + kOffV, sQ = sbase + kOffQ, sDO = sbase + kOffDO,
                 sDQ = sbase + kOffDQ, sDS = sbase + kOffDS;
  float* sL = reinterpret_cast<float*>(smem + kOffL);
  float* sD = reinterpret_cast<float*>(smem + kOffD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  auto bar = [&](int i) { return tc::smem_u32(bars + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * B_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * B_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdArgs& a = p.a;
  const int64_t S = a.seqlen;

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == B_PFULL || i == B_DSFULL || i == B_LDEMPTY0 || i == B_LDEMPTY1) cnt = 256;
      if (i == B_DQCONS) cnt = 128;
      if (i == B_LDFULL0 || i == B_LDFULL1) cnt = 32;
      tc::mbar_init(bar(i), cnt);
    }
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
  const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  // this CTA's work indices (planner schedule, head-major)
  const int32_t k_begin = a.kv_cta[blockIdx.x], k_end = a.kv_cta[blockIdx.x + 1];

  if (warp < 4) {
    tc::setmaxnreg_dec<kSmallRegs>();
  }
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&p.tmq);
      tc::prefetch_tmap(&p.tmk);
      tc::prefetch_tmap(&p.tmv);
      tc::prefetch_tmap(&p.tmdo);
      // loads armed per barrier (scalars: a runtime-indexed array would live in
      // local memory, whose accesses queue behind the dQ reductions)
      uint32_t gt = 0, ni = 0, armed_kv = 0, armed_q0 = 0, armed_q1 = 0, armed_do = 0;
      bool ok = true;
      for (int32_t kw = k_begin; kw < k_end && ok; ++kw) {
        const Item it = load_item(p, a.kv_work[kw]);
        if (it.n_tiles == 0) continue;
        const int rbase = int(int64_t(it.b) * S);
        ok = tc::wait_bounded<kShortWaits>(bar(B_KVEMPTY), (ni & 1) ^ 1, abort_flag, p.err, p.wait_limit);
        ++ni;
        if (!ok) break;
        tc::mbar_arrive_expect_tx(bar(B_KVFULL), 2 * kTileBytes);
        tc::tma_load_3d(sK, &p.tmk, bar(B_KVFULL), 0, it.g, rbase + it.row0);
        tc::tma_load_3d(sK + kHalfBytes, &p.tmk, bar(B_KVFULL), 64, it.g, rbase + it.row0);
        tc::tma_load_3d(sV, &p.tmv, bar(B_KVFULL), 0, it.g, rbase + it.row0);
        tc::tma_load_3d(sV + kHalfBytes, &p.tmv, bar(B_KVFULL), 64, it.g, rbase + it.row0);
        ++armed_kv;
        Walk wk = walk_begin(a, it);
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
          const QTile qt = walk_tile(a, it, wk);
          const uint32_t st = gt & 1, ph = (gt >> 1) & 1;
          ok = tc::wait_bounded<kShortWaits>(bar(B_QEMPTY0 + st), ph ^ 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          KV_TRACE(14, gt);
          tc::mbar_arrive_expect_tx(bar(B_QFULL0 + st), kTileBytes);
          tc::tma_load_3d(sQ + st * kTileBytes, &p.tmq, bar(B_QFULL0 + st), 0, qt.h, rbase + qt.q0);
          tc::tma_load_3d(sQ + st * kTileBytes + kHalfBytes, &p.tmq, bar(B_QFULL0 + st), 64, qt.h, rbase + qt.q0);
          if (st) ++armed_q1; else ++armed_q0;
          // one dO stage: dO(t) once dV(t-1) and dP(t-1) have read dO(t-1)
          ok = tc::wait_bounded<kShortWaits>(bar(B_DOEMPTY), (gt & 1) ^ 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(bar(B_DOFULL), kTileBytes);
          tc::tma_load_3d(sDO, &p.tmdo, bar(B_DOFULL), 0, qt.h, rbase + qt.q0);
          tc::tma_load_3d(sDO + kHalfBytes, &p.tmdo, bar(B_DOFULL), 64, qt.h, rbase + qt.q0);
          ++armed_do;
        }
      }
      volatile int never = 0;
      if (armed_kv) tc::mbar_wait(bar(B_KVFULL), (armed_kv - 1) & 1, &never, nullptr);
      for (int s = 0; s < 2; ++s) {
        const uint32_t nq = s ? armed_q1 : armed_q0;
        if (nq) tc::mbar_wait(bar(B_QFULL0 + s), (nq - 1) & 1, &never, nullptr);
      }
      if (armed_do) tc::mbar_wait(bar(B_DOFULL), (armed_do - 1) & 1, &never, nullptr);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t gt = 0, ni = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t g) {  // S^T = K Q^T
        const uint32_t q_s = sQ + (g & 1) * kTileBytes;
        const uint64_t a0 = opaque(tc::kmajor_desc(sK)), b0 = opaque(tc::kmajor_desc(q_s));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_ss(tS, tc::kmajor_step(a0, kk), tc::kmajor_step(b0, kk), kIdescKK, kk > 0);
        tc::mma_commit(bar(B_SFULL));
        KV_TRACE(0, g);
      };
      auto issue_dp = [&](uint32_t g) {  // dP^T = V dO^T
        const uint64_t a0 = opaque(tc::kmajor_desc(sV)), b0 = opaque(tc::kmajor_desc(sDO));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_ss(tDP, tc::kmajor_step(a0, kk), tc::kmajor_step(b0, kk), kIdescKK, kk > 0);
        tc::mma_commit(bar(B_DPFULL));
        KV_TRACE(4, g);
      };
      for (int32_t kw = k_begin; kw < k_end && ok; ++kw) {
        const Item it = load_item(p, a.kv_work[kw]);
        if (it.n_tiles == 0) continue;
        ok = tc::wait_bounded<kShortWaits>(bar(B_KVFULL), ni & 1, abort_flag, p.err, p.wait_limit);
        ++ni;
        // S of the item's first tile once dV of the previous tile has read P^T
        if (ok) ok = tc::wait_bounded<kShortWaits>(bar(B_QFULL0 + (gt & 1)), (gt >> 1) & 1, abort_flag, p.err, p.wait_limit);
        if (ok && gt > 0) ok = tc::wait_bounded<kShortWaits>(bar(B_PCONS), (gt - 1) & 1, abort_flag, p.err, p.wait_limit);
        if (!ok) break;
        tc::fence_after_sync();
        issue_s(gt);
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt) {
          const uint32_t st = gt & 1;
          const bool has_next = t + 1 < it.n_tiles;
          // dP^T into the columns of the previous tile's dQ once it is read
          // out: it needs no P, so it runs while the math warps build P^T
          ok = tc::wait_bounded<kShortWaits>(bar(B_DOFULL), gt & 1, abort_flag, p.err, p.wait_limit);
          if (ok && gt > 0)
            ok = tc::wait_bounded<kShortWaits>(bar(B_DQCONS), (gt - 1) & 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          KV_TRACE(3, gt);
          tc::fence_after_sync();
          issue_dp(gt);
          ok = tc::wait_bounded<kShortWaits>(bar(B_PFULL), gt & 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          KV_TRACE(1, gt);
          tc::fence_after_sync();
          const uint64_t bv = opaque(tc::mnmajor_desc(sDO));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO, P^T from TMEM
            tc::mma_ts(tDV, tS + (kk >> 2) * 64 + (kk & 3) * 8, tc::mnmajor_step(bv, kk), kIdescKM,
                       (t > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(bar(B_PCONS));
          tc::mma_commit(bar(B_DOEMPTY));  // dP and dV have read dO
          KV_TRACE(2, gt);
          if (has_next) {  // S of the next tile once dV has read P^T
            ok = tc::wait_bounded<kShortWaits>(bar(B_QFULL0 + (st ^ 1)), ((gt + 1) >> 1) & 1, abort_flag, p.err, p.wait_limit) &&
                 tc::wait_bounded<kShortWaits>(bar(B_PCONS), gt & 1, abort_flag, p.err, p.wait_limit);
            if (!ok) break;
            tc::fence_after_sync();
            issue_s(gt + 1);
          }
          ok = tc::wait_bounded<kShortWaits>(bar(B_DSFULL), gt & 1, abort_flag, p.err, p.wait_limit);
          if (!ok) break;
          KV_TRACE(5, gt);
          tc::fence_after_sync();
          // dQ first: its read-out (which frees the dP^T columns for the next
          // tile's dP) overlaps dK on the tensor core
          const uint64_t aq = opaque(tc::mnmajor_desc(sDS)), bq = opaque(tc::mnmajor_desc(sK));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ_t = dS K over the dP^T columns (read out by the dQ warps)
            tc::mma_ss(tDP, tc::mnmajor_step(aq, kk), tc::mnmajor_step(bq, kk), kIdescMM, kk > 0 ? 1u : 0u);
          tc::mma_commit(bar(B_DQFULL));
          const uint64_t ak = opaque(tc::kmajor_desc(sDS)), bk = opaque(tc::mnmajor_desc(sQ + st * kTileBytes));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q
            tc::mma_ss(tDK, tc::kmajor_step(ak, kk), tc::mnmajor_step(bk, kk), kIdescKM, (t > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(bar(B_QEMPTY0 + st));
          KV_TRACE(6, gt);
          if (!has_next) {
            tc::mma_commit(bar(B_KVEMPTY));
            tc::mma_commit(bar(B_DKDV));
          }
        }
      }
      volatile int never = 0;
      tc::mma_commit(bar(B_DRAIN));
      tc::mbar_wait(bar(B_DRAIN), 0, &never, nullptr);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------- key-row math warps --
    // Eight warps, two per TMEM lane quarter: warp w serves key rows
    // 32 (w % 4) .. +31 and query columns 64 h .. 64 h + 63, h = (w - 4) / 4.
    tc::setmaxnreg_inc<kMathRegs>();
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int j = quarter * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t gt = 0, ni = 0;
    bool ok = true;
    for (int32_t kw = k_begin; kw < k_end && ok; ++kw) {
      const Item it = load_item(p, a.kv_work[kw]);
      const bool kvalid = j < it.len;
      const int kpos = it.pos0 + j;
      if (it.n_tiles > 0) {
        Walk wk = walk_begin(a, it);
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
          const QTile qt = walk_tile(a, it, wk);
          const uint32_t st = gt & 1;
          ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_LDFULL0 + st), (gt >> 1) & 1, abort_flag, p.err, p.wait_limit) &&
                                           tc::wait_bounded<kShortWaits>(bar(B_SFULL), gt & 1, abort_flag, p.err, p.wait_limit));
          if (!ok) break;
          if (warp == 4 && lane == 0) KV_TRACE(7, gt);
          tc::fence_after_sync();
          // visible queries: i_lo <= i < i_hi (i_hi < kTile only under a
          // sliding window; queries past the tile have -L2 = -inf)
          int i_lo = a.causal ? max(0, kpos - qt.qpos0) : 0;
          if (!kvalid) i_lo = kTile;
          const int i_hi = qt.win > 0 ? kpos + qt.win - qt.qpos0 : kTile;
          const bool open = __all_sync(0xffffffffu, i_lo <= half * 64 && i_hi >= half * 64 + 64);  // no masking
          const uint32_t i_span = uint32_t(max(min(i_hi, kTile) - i_lo, 0));
          const float4* L4 = reinterpret_cast<const float4*>(sL + st * 128 + half * 64);  // -L2
          const float4* D4 = reinterpret_cast<const float4*>(sD + st * 128 + half * 64);  // -D
          const uint64_t sl2x2 = tc::f32x2(sl2, sl2);
          uint32_t pk[32];
          uint32_t sr64[64];
          tc::tmem_ld32(tS + lane_off + half * 64, sr64);
          tc::tmem_ld32(tS + lane_off + half * 64 + 32, sr64 + 32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {  // P^T = exp2(S^T sl2 - L2); P^T kept in its own half
            const uint32_t* sr = sr64 + cc * 32;
            const int col0 = half * 64 + cc * 32;
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 l4 = L4[cc * 8 + e4];
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const int e = e4 * 2 + e2;
                float x0, x1;
                tc::f32x2_split(tc::ffma2(tc::f32x2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])),
                                          sl2x2, tc::f32x2(lv[2 * e2], lv[2 * e2 + 1])),
                                x0, x1);
                pk[cc * 16 + e] = tc::pack_bf16x2(tc::ex2(x0), tc::ex2(x1));
              }
            }
            if (!open) {  // clear the invisible pairs' bf16 halves (an overflowed exp becomes 0 too)
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int i0 = col0 + 2 * e;
                const uint32_t keep = (uint32_t(i0 - i_lo) < i_span ? 0x0000ffffu : 0u) |
                                      (uint32_t(i0 + 1 - i_lo) < i_span ? 0xffff0000u : 0u);
                pk[cc * 16 + e] &= keep;
              }
            }
            tc::tmem_st16(tS + lane_off + half * 64 + cc * 16, pk + cc * 16);
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
          tc::mbar_arrive(bar(B_PFULL));
          if (warp == 4 && lane == 0) KV_TRACE(8, gt);
          ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_DPFULL), gt & 1, abort_flag, p.err, p.wait_limit));
          if (!ok) break;
          if (warp == 4 && lane == 0) KV_TRACE(12, gt);
          tc::fence_after_sync();
          uint32_t dr64[64];
          tc::tmem_ld32(tDP + lane_off + half * 64, dr64);
          tc::tmem_ld32(tDP + lane_off + half * 64 + 32, dr64 + 32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {  // dS^T = P^T (dP^T - D)
            const uint32_t* dr = dr64 + cc * 32;
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 d4 = D4[cc * 8 + e4];
              const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const int e = e4 * 2 + e2;
                const uint32_t w2 = pk[cc * 16 + e];
                const uint64_t dd = tc::fadd2(tc::f32x2(__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])),
                                              tc::f32x2(dv4[2 * e2], dv4[2 * e2 + 1]));
                float d0, d1;
                tc::f32x2_split(tc::fmul2(tc::f32x2(__uint_as_float(w2 << 16), __uint_as_float(w2 & 0xFFFF0000u)), dd),
                                d0, d1);
                pk[cc * 16 + e] = tc::pack_bf16x2(d0, d1);
              }
            }
          }
          tc::fence_before_sync();
          tc::mbar_arrive(bar(B_LDEMPTY0 + st));
          // dK and dQ of the previous tile (issued before this dP) have read the old dS^T;
          // this warp writes its 64 query columns = one 128-byte swizzle region
          uint8_t* drow = smem + kOffDS + half * kHalfBytes + j * 128;
#pragma unroll
          for (int kc = 0; kc < 8; ++kc)
            *reinterpret_cast<uint4*>(drow + ((kc ^ (j & 7)) << 4)) =
                make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
          tc::fence_proxy_async_smem();
          tc::fence_before_sync();
          tc::mbar_arrive(bar(B_DSFULL));
          if (warp == 4 && lane == 0) KV_TRACE(13, gt);
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_DKDV), ni & 1, abort_flag, p.err, p.wait_limit));
        ++ni;
        if (!ok) break;
        tc::fence_after_sync();
      }
      // item epilogue: half 0 writes dV, half 1 writes scale * dK of this key row
      const int64_t orow = ((int64_t(it.b) * S + it.row0 + j) * a.Hkv + it.g) * 128;
      const uint32_t tsrc = half == 0 ? tDV : tDK;
      const float mul = half == 0 ? 1.f : a.scale;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(half == 0 ? a.dv : a.dk) + orow;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        if (it.n_tiles > 0) {
          tc::tmem_ld32(tsrc + lane_off + c * 32, r);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        if (kvalid) store_row_bf16(dst + c * 32, r, mul);
      }
      tc::fence_before_sync();
    }
  } else if (warp == 2) {
    // ---------------------------------------------- L and D staging warp --
    uint32_t gt = 0;
    bool ok = true;
    for (int32_t kw = k_begin; kw < k_end && ok; ++kw) {
      const Item it = load_item(p, a.kv_work[kw]);
      if (it.n_tiles == 0) continue;
      Walk wk = walk_begin(a, it);
      for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
        const QTile qt = walk_tile(a, it, wk);
        const uint32_t st = gt & 1;
        ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_LDEMPTY0 + st), ((gt >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_limit));
        if (!ok) break;
        const int64_t base = (int64_t(it.b) * a.H + qt.h) * S + qt.q0;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int q = lane + 32 * k4;
          const bool v = q < qt.qlen;
          sL[st * 128 + q] = v ? -a.lse2[base + q] : -INFINITY;  // -L2: exp2(S sl2 - L2) = 0 past the tile
          sD[st * 128 + q] = v ? -a.delta[base + q] : 0.f;
        }
        tc::mbar_arrive(bar(B_LDFULL0 + st));
        if (lane == 0) KV_TRACE(15, gt);
      }
    }
  } else if (warp >= 12) {
    // --------------------------------------------- dQ read-out warps --
    // Warp w reads TMEM lane quarter w % 4 = query rows 32 (w % 4) .. +31 of
    // the tile, all 128 dQ columns, and hands the columns back for the next
    // dP^T.  The four warps then stage the tile in 32-column chunks (two
    // staging buffers) and one thread adds each chunk into the accumulator
    // with a TMA reduction.  Named barrier 1 orders the four warps; the
    // tile's wait result is agreed on at that barrier, so a wait that gives
    // up stops all four together.
    tc::setmaxnreg_inc<kDqRegs>();
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const bool leader = warp == 12 && lane == 0;
    if (leader) tc::prefetch_tmap(&p.tmdq);
    uint32_t gt = 0, nchunk = 0;
    bool ok = true;
    for (int32_t kw = k_begin; kw < k_end && ok; ++kw) {
      const Item it = load_item(p, a.kv_work[kw]);
      if (it.n_tiles == 0) continue;
      Walk wk = walk_begin(a, it);
      for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
        const QTile qt = walk_tile(a, it, wk);
        ok = __all_sync(0xffffffffu, tc::wait_bounded<kShortWaits>(bar(B_DQFULL), gt & 1, abort_flag, p.err, p.wait_limit));
        ok = tc::named_bar_all(1, 128, ok);
        if (!ok) break;
        if (quarter == 0 && lane == 0) KV_TRACE(9, gt);
        tc::fence_after_sync();
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(tDP + lane_off + c * 32, r + c * 32);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        tc::mbar_arrive(bar(B_DQCONS));
        if (quarter == 0 && lane == 0) KV_TRACE(10, gt);
        const int plane = it.b * a.H + qt.h;
#pragma unroll
        for (int c = 0; c < 4; ++c, ++nchunk) {
          const uint32_t buf = sDQ + (nchunk & 1) * kDqChunkBytes;
          if (leader && nchunk >= 2) tc::bulk_wait_group_read<1>();  // the reduction that last used buf has read it
          tc::named_bar(1, 128);
          // row i: 32 floats = 8 x 16 bytes, 128-byte swizzle (unit k at k ^ (i % 8))
          uint8_t* row = smem + (buf - sbase) + i * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(row + ((k ^ (i & 7)) << 4)) =
                make_uint4(r[32 * c + 4 * k], r[32 * c + 4 * k + 1], r[32 * c + 4 * k + 2], r[32 * c + 4 * k + 3]);
          tc::fence_proxy_async_smem();
          tc::named_bar(1, 128);
          if (leader) {
            tc::tma_reduce_add_3d(&p.tmdq, buf, c * 32, qt.q0, plane);
            tc::bulk_commit_group();
          }
        }
        if (quarter == 0 && lane == 0) KV_TRACE(11, gt);
      }
    }
    if (leader) tc::bulk_wait_group<0>();  // every reduction complete before the block exits
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace kv

// ====================================================== dQ conversion ======
// dQ = scale * accumulator: the accumulator as a flat array of float4, 32 per
// (batch * q-head, row); a warp's 32 consecutive float4 are one row (512 bytes
// read, 256 bytes written), and each thread converts four of them per step so
// that four loads are in flight.
__global__ void __launch_bounds__(256) dq_post_kernel(const float4* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                      int64_t S, int H, int64_t n4, float scale) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n4; i0 += 4 * stride) {
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      x[u] = i < n4 ? acc[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= n4) break;
      const int64_t row = i >> 5;
      const int64_t bh = row / S, srow = row - bh * S;
      const int64_t b = bh / H, h = bh - b * H;
      uint2 v;
      v.x = tc::pack_bf16x2(x[u].x * scale, x[u].y * scale);
      v.y = tc::pack_bf16x2(x[u].z * scale, x[u].w * scale);
      *reinterpret_cast<uint2*>(dq + ((b * S + srow) * H + h) * 128 + (i & 31) * 4) = v;
    }
  }
}

// Raises the kernel's dynamic shared memory limit once per device (setting it
// again from a racing host thread is harmless).
template <typename K>
cp_status set_smem(K kernel, int bytes, std::atomic<bool>* done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return CP_ERR_CUDA;
    done[dev].store(true, std::memory_order_release);
  }
  return CP_OK;
}

}  // namespace

#ifdef CPATTN_TRACE
extern "C" int cp_kv_trace_dump(unsigned long long* out, int max_events) {
  cudaDeviceSynchronize();
  const int n = max_events < kv::kTraceEvents * kv::kTraceTiles ? max_events : kv::kTraceEvents * kv::kTraceTiles;
  cudaMemcpyFromSymbol(out, kv::g_kv_trace, sizeof(unsigned long long) * n);
  return n;
}
#endif

cp_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
  static std::atomic<bool> kv_set[2][64] = {};
  if (!a.dq_acc) return CP_ERR_INVALID_ARG;
  if (a.dtype != CP_BF16 || a.d != 128) return CP_ERR_UNSUPPORTED;
  const long long limit = wait_limit_cycles();
  const bool short_waits = limit < tc::kWaitCycles;
  auto* kern = short_waits ? kv::dkdv_kernel<true> : kv::dkdv_kernel<false>;
  {
    // The register hand-over inside the kernel assumes the launch count.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return CP_ERR_CUDA;
    if (fa.numRegs != kv::kLaunchRegs) return CP_ERR_UNSUPPORTED;
  }
  cp_status st = set_smem(kern, kv::kSmemBytes, kv_set[short_waits]);
  if (st != CP_OK) return st;
  Params p;
  const int64_t rows = int64_t(a.batch) * a.seqlen;
  if (!make_tmap_rows(&p.tmq, a.q, rows, a.H, 128, 128) ||
      !make_tmap_rows(&p.tmk, a.k, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmv, a.v, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmdo, a.dout, rows, a.H, 128, 128) ||
      !make_tmap_f32_chunks(&p.tmdq, a.dq_acc, int64_t(a.batch) * a.H, a.seqlen))
    return CP_ERR_CUDA;
  p.a = a;
  p.err = device_error_ptr();
  p.wait_limit = limit;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (a.n_kv_items > 0 && a.kv_grid > 0) {
    kern<<<unsigned(a.kv_grid), kv::kThreads, kv::kSmemBytes, s>>>(p);
    st = cuda_status(cudaGetLastError());
    if (st != CP_OK) return st;
  }
  return st;
}

cp_status launch_dq_post(const BwdArgs& a, cudaStream_t s) {
  if (!a.dq_acc) return CP_ERR_INVALID_ARG;
  const int64_t n4 = int64_t(a.batch) * a.H * a.seqlen * 32;
  if (n4 == 0) return CP_OK;
  int64_t grid = (n4 + 1023) / 1024;  // four float4 per thread and step
  const int64_t cap = int64_t(num_sms()) * 8;
  grid = grid < cap ? grid : cap;
  dq_post_kernel<<<unsigned(grid), 256, 0, s>>>(reinterpret_cast<const float4*>(a.dq_acc),
                                                static_cast<__nv_bfloat16*>(a.dq), a.seqlen, a.H, n4, a.scale);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
