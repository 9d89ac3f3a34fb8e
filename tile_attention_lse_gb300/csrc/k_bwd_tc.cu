// tcgen05 tile-attention backward for bf16, head_dim 128 (sm_103a).
//
// "上下文并行" 01 BACKWARD/REPLAY and GRADIENT/RETURN: every block of the
// task graph is replayed from the merged row LSE (P = exp(S - L), no second
// softmax pass) and D = <dO, O>; with dS = P (dP - D) the block contributes
//   dV_j += sum_i P_ij dO_i,  dK_j += scale sum_i dS_ij Q_i,
//   dQ_i += scale sum_j dS_ij K_j.
// A work item is one K/V tile (128 keys of one kv-head) together with every Q
// range of every query rank that sees it (in ring order) and every q-head of
// the group: the dK/dV contributions of all query ranks are summed in TMEM at
// the key owner and written once.  dQ tiles are accumulated into a float32
// buffer with vector reductions.
//
// Persistent kernel, one CTA per SM, 352 threads:
//   warp 0      TMA producer: K and V once per item, Q and dO per query tile
//               (2-stage rings of 128-byte-swizzled 64 x 128 boxes);
//   warp 1      tcgen05.mma issuer and TMEM owner.  Per query tile:
//                 S^T  = K Q^T        -> TMEM [0,128)   (keys on lanes)
//                 dP^T = V dO^T       -> TMEM [128,256)
//                 dV  += P^T dO       -> TMEM [256,384) (dO read MN-major)
//                 dK  += dS^T Q       -> TMEM [384,512) (Q read MN-major)
//                 dQ   = dS K         -> TMEM [0,128)   (dS^T read MN-major)
//   warps 2..5  key-row math: P^T = exp2(S^T log2e*scale - L log2e) with the
//               causal mask by original position, dS^T = P^T (dP^T - D); both
//               written as bf16 to one shared tile in the MMA's K-major layout;
//               at the end of an item dK (times scale) and dV to global, bf16;
//   warps 6..9  dQ drain: TMEM -> red.global.add.v4.f32 (times scale);
//   warp 10     stages L*log2e and D of each query tile into shared memory.
// Every mbarrier wait is bounded (device error word + orderly exit).
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace cpattn {

namespace {

constexpr int kThreads = 352;
constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;        // 2 stages
constexpr int kOffDO = kOffQ + 2 * kTileBytes;   // 2 stages
constexpr int kOffPdS = kOffDO + 2 * kTileBytes;
constexpr int kOffL = kOffPdS + kTileBytes;      // 2 stages x 128 floats
constexpr int kOffD = kOffL + 2 * 512;           // 2 stages x 128 floats
constexpr int kOffBar = kOffD + 2 * 512;
constexpr int kSmemBytes = kOffBar + 256;

enum {
  B_KVFULL = 0, B_KVEMPTY, B_QFULL0, B_QFULL1, B_QEMPTY0, B_QEMPTY1, B_DOFULL0, B_DOFULL1,
  B_DOEMPTY0, B_DOEMPTY1, B_SFULL, B_DPFULL, B_PFULL, B_PCONS, B_DSFULL, B_PDSFREE, B_DQFULL,
  B_DQFREE, B_DKDV, B_LDFULL0, B_LDFULL1, B_LDEMPTY0, B_LDEMPTY1, B_DRAIN, B_COUNT
};
static_assert(kOffBar + 8 * B_COUNT + 8 <= kSmemBytes, "barrier area");

constexpr uint32_t kIdescKK = tc::idesc_bf16(128, 128, 0, 0);  // A, B K-major
constexpr uint32_t kIdescKM = tc::idesc_bf16(128, 128, 1, 0);  // B MN-major
constexpr uint32_t kIdescMM = tc::idesc_bf16(128, 128, 1, 1);  // A, B MN-major

struct Params {
  CUtensorMap tmq, tmk, tmv, tmdo;
  BwdArgs a;
  int* err;
  float scale_log2;
  int64_t total_work;
};

struct KvItem {
  int32_t row0, pos0, len, seg_begin, seg_count;
  int b, g;
  int n_tiles;  // query tiles over all q-heads of the group
};

__device__ __forceinline__ KvItem load_kv_item(const Params& p, int64_t w) {
  const BwdArgs& a = p.a;
  const int64_t bh = w / a.n_kv_items;
  const int idx = int(w - bh * a.n_kv_items);
  KvItem it;
  it.b = int(bh / a.Hkv);
  it.g = int(bh - int64_t(it.b) * a.Hkv);
  const TileItem t = a.kv_items[idx];
  it.row0 = t.row0;
  it.pos0 = t.pos0;
  it.len = t.len;
  it.seg_begin = t.seg_begin;
  it.seg_count = t.seg_count;
  int n = 0;
  for (int s = 0; s < t.seg_count; ++s) n += (a.kv_segs[t.seg_begin + s].len + kTile - 1) / kTile;
  it.n_tiles = n * (a.H / a.Hkv);
  return it;
}

// Walks the query tiles of an item: q-head of the group, then segment, then
// 128-row tile.  Every role advances an identical walker.
struct QWalk {
  int hj, si, u;
};

struct QTile {
  int h, q0, qpos0, qlen;
};

__device__ __forceinline__ QTile walk_tile(const BwdArgs& a, const KvItem& it, const QWalk& w) {
  const Seg sg = a.kv_segs[it.seg_begin + w.si];
  QTile t;
  t.h = it.g * (a.H / a.Hkv) + w.hj;
  t.q0 = sg.row0 + w.u * kTile;
  t.qpos0 = sg.pos0 + w.u * kTile;
  t.qlen = min(kTile, sg.len - w.u * kTile);
  return t;
}

__device__ __forceinline__ void walk_next(const BwdArgs& a, const KvItem& it, QWalk& w) {
  const Seg sg = a.kv_segs[it.seg_begin + w.si];
  if ((w.u + 1) * kTile < sg.len) {
    ++w.u;
    return;
  }
  w.u = 0;
  // skip empty segments
  do {
    ++w.si;
    if (w.si == it.seg_count) {
      w.si = 0;
      ++w.hj;
    }
  } while (w.hj < a.H / a.Hkv && a.kv_segs[it.seg_begin + w.si].len <= 0);
}

__device__ __forceinline__ QWalk walk_begin(const BwdArgs& a, const KvItem& it) {
  QWalk w{0, 0, 0};
  while (w.si < it.seg_count && a.kv_segs[it.seg_begin + w.si].len <= 0) ++w.si;
  return w;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = tc::smem_u32(smem);
  if (sbase & 1023) {  // the swizzled layouts need a 1 KB aligned base
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 2);
    return;
  }
  const uint32_t sK = sbase + kOffK, sV = sbase + kOffV, sQ = sbase + kOffQ, sDO = sbase + kOffDO,
                 sPdS = sbase + kOffPdS;
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
      if (i == B_PFULL || i == B_DSFULL || i == B_DQFREE || i == B_LDEMPTY0 || i == B_LDEMPTY1) cnt = 128;
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
  const int64_t first = blockIdx.x, stride = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&p.tmq);
      tc::prefetch_tmap(&p.tmk);
      tc::prefetch_tmap(&p.tmv);
      tc::prefetch_tmap(&p.tmdo);
      uint32_t gt = 0, ni = 0, armed_kv = 0, armed_q[2] = {0, 0}, armed_do[2] = {0, 0};
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        const KvItem it = load_kv_item(p, w);
        if (it.n_tiles == 0) continue;
        const int rbase = int(int64_t(it.b) * S);
        ok = tc::mbar_wait(bar(B_KVEMPTY), (ni & 1) ^ 1, abort_flag, p.err);
        ++ni;
        if (!ok) break;
        tc::mbar_arrive_expect_tx(bar(B_KVFULL), 2 * kTileBytes);
        tc::tma_load_3d(sK, &p.tmk, bar(B_KVFULL), 0, it.g, rbase + it.row0);
        tc::tma_load_3d(sK + kHalfBytes, &p.tmk, bar(B_KVFULL), 64, it.g, rbase + it.row0);
        tc::tma_load_3d(sV, &p.tmv, bar(B_KVFULL), 0, it.g, rbase + it.row0);
        tc::tma_load_3d(sV + kHalfBytes, &p.tmv, bar(B_KVFULL), 64, it.g, rbase + it.row0);
        ++armed_kv;
        QWalk wk = walk_begin(a, it);
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
          const QTile qt = walk_tile(a, it, wk);
          const uint32_t st = gt & 1, ph = (gt >> 1) & 1;
          ok = tc::mbar_wait(bar(B_QEMPTY0 + st), ph ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(bar(B_QFULL0 + st), kTileBytes);
          tc::tma_load_3d(sQ + st * kTileBytes, &p.tmq, bar(B_QFULL0 + st), 0, qt.h, rbase + qt.q0);
          tc::tma_load_3d(sQ + st * kTileBytes + kHalfBytes, &p.tmq, bar(B_QFULL0 + st), 64, qt.h, rbase + qt.q0);
          ++armed_q[st];
          ok = tc::mbar_wait(bar(B_DOEMPTY0 + st), ph ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(bar(B_DOFULL0 + st), kTileBytes);
          tc::tma_load_3d(sDO + st * kTileBytes, &p.tmdo, bar(B_DOFULL0 + st), 0, qt.h, rbase + qt.q0);
          tc::tma_load_3d(sDO + st * kTileBytes + kHalfBytes, &p.tmdo, bar(B_DOFULL0 + st), 64, qt.h, rbase + qt.q0);
          ++armed_do[st];
        }
      }
      volatile int never = 0;
      if (armed_kv) tc::mbar_wait(bar(B_KVFULL), (armed_kv - 1) & 1, &never, nullptr);
      for (int s = 0; s < 2; ++s) {
        if (armed_q[s]) tc::mbar_wait(bar(B_QFULL0 + s), (armed_q[s] - 1) & 1, &never, nullptr);
        if (armed_do[s]) tc::mbar_wait(bar(B_DOFULL0 + s), (armed_do[s] - 1) & 1, &never, nullptr);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t gt = 0, ni = 0;
      bool ok = true;
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        const KvItem it = load_kv_item(p, w);
        if (it.n_tiles == 0) continue;
        ok = tc::mbar_wait(bar(B_KVFULL), ni & 1, abort_flag, p.err);
        ++ni;
        if (!ok) break;
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt) {
          const uint32_t st = gt & 1, ph = (gt >> 1) & 1;
          ok = tc::mbar_wait(bar(B_QFULL0 + st), ph, abort_flag, p.err) &&
               tc::mbar_wait(bar(B_DOFULL0 + st), ph, abort_flag, p.err);
          if (ok && gt > 0) ok = tc::mbar_wait(bar(B_DQFREE), (gt - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t q_s = sQ + st * kTileBytes, do_s = sDO + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // S^T = K Q^T
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            tc::mma_ss(tS, tc::smem_desc(sK + off, 16, 1024), tc::smem_desc(q_s + off, 16, 1024),
                       kIdescKK, kk > 0);
          }
          tc::mma_commit(bar(B_SFULL));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dP^T = V dO^T
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            tc::mma_ss(tDP, tc::smem_desc(sV + off, 16, 1024), tc::smem_desc(do_s + off, 16, 1024),
                       kIdescKK, kk > 0);
          }
          tc::mma_commit(bar(B_DPFULL));
          ok = tc::mbar_wait(bar(B_PFULL), gt & 1, abort_flag, p.err);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dV += P^T dO
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            tc::mma_ss(tDV, tc::smem_desc(sPdS + off, 16, 1024),
                       tc::smem_desc(do_s + kk * 2048, kHalfBytes, 1024), kIdescKM,
                       (t > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(bar(B_PCONS));
          tc::mma_commit(bar(B_DOEMPTY0 + st));
          ok = tc::mbar_wait(bar(B_DSFULL), gt & 1, abort_flag, p.err);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dK += dS^T Q
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            tc::mma_ss(tDK, tc::smem_desc(sPdS + off, 16, 1024),
                       tc::smem_desc(q_s + kk * 2048, kHalfBytes, 1024), kIdescKM,
                       (t > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dQ = dS K
            tc::mma_ss(tS, tc::smem_desc(sPdS + kk * 2048, kHalfBytes, 1024),
                       tc::smem_desc(sK + kk * 2048, kHalfBytes, 1024), kIdescMM, kk > 0);
          }
          tc::mma_commit(bar(B_QEMPTY0 + st));
          tc::mma_commit(bar(B_DQFULL));
          tc::mma_commit(bar(B_PDSFREE));
          if (t == it.n_tiles - 1) {
            tc::mma_commit(bar(B_KVEMPTY));
            tc::mma_commit(bar(B_DKDV));
          }
        }
      }
      volatile int never = 0;
      tc::mma_commit(bar(B_DRAIN));
      tc::mbar_wait(bar(B_DRAIN), 0, &never, nullptr);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------- key-row math warps --
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;  // key row in the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t gt = 0, ni = 0;
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      const KvItem it = load_kv_item(p, w);
      const bool kvalid = j < it.len;
      const int kpos = it.pos0 + j;
      if (it.n_tiles > 0) {
        QWalk wk = walk_begin(a, it);
        for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
          const QTile qt = walk_tile(a, it, wk);
          const uint32_t st = gt & 1;
          ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_LDFULL0 + st), (gt >> 1) & 1, abort_flag, p.err) &&
                                           tc::mbar_wait(bar(B_SFULL), gt & 1, abort_flag, p.err));
          if (!ok) break;
          tc::fence_after_sync();
          // queries i in [i_lo, qlen) are visible to this key
          int i_lo = a.causal ? max(0, kpos - qt.qpos0) : 0;
          if (!kvalid) i_lo = kTile;
          const float* Lst = sL + st * 128;
          const float* Dst = sD + st * 128;
          uint32_t pk[64];  // P^T row as bf16 pairs, later dS^T
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t sr[32];
            tc::tmem_ld32(tS + lane_off + c * 32, sr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int i0 = c * 32 + 2 * e;
              const float x0 = (i0 >= i_lo && i0 < qt.qlen) ? fmaf(__uint_as_float(sr[2 * e]), sl2, -Lst[i0]) : -INFINITY;
              const float x1 = (i0 + 1 >= i_lo && i0 + 1 < qt.qlen) ? fmaf(__uint_as_float(sr[2 * e + 1]), sl2, -Lst[i0 + 1]) : -INFINITY;
              pk[c * 16 + e] = tc::pack_bf16x2(tc::ex2(x0), tc::ex2(x1));
            }
          }
          if (gt > 0) {
            ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_PDSFREE), (gt - 1) & 1, abort_flag, p.err));
            if (!ok) break;
          }
          uint8_t* prow = smem + kOffPdS + j * 128;
#pragma unroll
          for (int kc = 0; kc < 16; ++kc) {
            const int region = kc >> 3, chunk = kc & 7;
            *reinterpret_cast<uint4*>(prow + region * kHalfBytes + ((chunk ^ (j & 7)) << 4)) =
                make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
          }
          tc::fence_proxy_async_smem();
          tc::fence_before_sync();
          tc::mbar_arrive(bar(B_PFULL));
          ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_DPFULL), gt & 1, abort_flag, p.err));
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t dr[32];
            tc::tmem_ld32(tDP + lane_off + c * 32, dr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int i0 = c * 32 + 2 * e;
              const uint32_t w2 = pk[c * 16 + e];
              const float p0 = __uint_as_float(w2 << 16), p1 = __uint_as_float(w2 & 0xFFFF0000u);
              const float d0 = p0 * (__uint_as_float(dr[2 * e]) - Dst[i0]);
              const float d1 = p1 * (__uint_as_float(dr[2 * e + 1]) - Dst[i0 + 1]);
              pk[c * 16 + e] = tc::pack_bf16x2(d0, d1);
            }
          }
          tc::fence_before_sync();
          // L and D of this stage are no longer needed
          tc::mbar_arrive(bar(B_LDEMPTY0 + st));
          ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_PCONS), gt & 1, abort_flag, p.err));
          if (!ok) break;
#pragma unroll
          for (int kc = 0; kc < 16; ++kc) {
            const int region = kc >> 3, chunk = kc & 7;
            *reinterpret_cast<uint4*>(prow + region * kHalfBytes + ((chunk ^ (j & 7)) << 4)) =
                make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
          }
          tc::fence_proxy_async_smem();
          tc::fence_before_sync();
          tc::mbar_arrive(bar(B_DSFULL));
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_DKDV), ni & 1, abort_flag, p.err));
        ++ni;
        if (!ok) break;
        tc::fence_after_sync();
      }
      // item epilogue: dV and scale * dK of this key row, bf16
      const int64_t orow = ((int64_t(it.b) * S + it.row0 + j) * a.Hkv + it.g) * 128;
      __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(a.dv) + orow;
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(a.dk) + orow;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t tsrc = which == 0 ? tDV : tDK;
        const float mul = which == 0 ? 1.f : a.scale;
        __nv_bfloat16* dst = which == 0 ? dvp : dkp;
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
          if (kvalid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 0]) * mul, __uint_as_float(r[8 * q4 + 1]) * mul);
              v.y = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 2]) * mul, __uint_as_float(r[8 * q4 + 3]) * mul);
              v.z = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 4]) * mul, __uint_as_float(r[8 * q4 + 5]) * mul);
              v.w = tc::pack_bf16x2(__uint_as_float(r[8 * q4 + 6]) * mul, __uint_as_float(r[8 * q4 + 7]) * mul);
              *reinterpret_cast<uint4*>(dst + c * 32 + q4 * 8) = v;
            }
          }
        }
      }
      tc::fence_before_sync();
    }
  } else if (warp >= 6 && warp <= 9) {
    // ------------------------------------------------------- dQ drain warps --
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    uint32_t gt = 0;
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      const KvItem it = load_kv_item(p, w);
      if (it.n_tiles == 0) continue;
      QWalk wk = walk_begin(a, it);
      for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
        const QTile qt = walk_tile(a, it, wk);
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_DQFULL), gt & 1, abort_flag, p.err));
        if (!ok) break;
        tc::fence_after_sync();
        const bool valid = i < qt.qlen;
        float* dst = a.dq_acc + ((int64_t(it.b) * S + qt.q0 + i) * a.H + qt.h) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tS + lane_off + c * 32, r);
          tc::tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              red_add_v4(dst + c * 32 + q4 * 4, __uint_as_float(r[4 * q4]) * a.scale,
                         __uint_as_float(r[4 * q4 + 1]) * a.scale, __uint_as_float(r[4 * q4 + 2]) * a.scale,
                         __uint_as_float(r[4 * q4 + 3]) * a.scale);
          }
        }
        tc::fence_before_sync();
        tc::mbar_arrive(bar(B_DQFREE));
      }
    }
  } else if (warp == 10) {
    // ---------------------------------------------- L and D staging warp --
    uint32_t gt = 0;
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      const KvItem it = load_kv_item(p, w);
      if (it.n_tiles == 0) continue;
      QWalk wk = walk_begin(a, it);
      for (int t = 0; t < it.n_tiles && ok; ++t, ++gt, walk_next(a, it, wk)) {
        const QTile qt = walk_tile(a, it, wk);
        const uint32_t st = gt & 1;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_LDEMPTY0 + st), ((gt >> 1) & 1) ^ 1, abort_flag, p.err));
        if (!ok) break;
        const int64_t base = (int64_t(it.b) * a.H + qt.h) * S + qt.q0;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int q = lane + 32 * k4;
          const bool v = q < qt.qlen;
          sL[st * 128 + q] = v ? a.lse2[base + q] : INFINITY;
          sD[st * 128 + q] = v ? a.delta[base + q] : 0.f;
        }
        tc::mbar_arrive(bar(B_LDFULL0 + st));
      }
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

bool bwd_tc_supported(const BwdArgs& a) {
  return a.dtype == CP_BF16 && a.d == 128 && tmap_encoder() != nullptr;
}

cp_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s) {
  if (a.n_kv_items == 0) return CP_OK;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return CP_ERR_CUDA;
    attr_set[dev] = true;
  }
  Params p;
  const int64_t rows = int64_t(a.batch) * a.seqlen;
  if (!make_tmap_rows(&p.tmq, a.q, rows, a.H, 128, 128) ||
      !make_tmap_rows(&p.tmk, a.k, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmv, a.v, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmdo, a.dout, rows, a.H, 128, 128))
    return CP_ERR_CUDA;
  p.a = a;
  p.err = device_error_ptr();
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.total_work = int64_t(a.n_kv_items) * a.batch * a.Hkv;
  const int64_t grid = p.total_work < num_sms() ? p.total_work : num_sms();
  bwd_tc_kernel<<<unsigned(grid), kThreads, kSmemBytes, s>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
