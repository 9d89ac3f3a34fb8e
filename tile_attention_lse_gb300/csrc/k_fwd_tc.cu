// tcgen05 tile-attention forward for bf16, head_dim 128 (sm_103a).
//
// Computes, for every work item (a tile of <= 128 queries and the K/V
// segments of one key owner: one edge of the task graph, "Context
// Parallelism (CP)" §2.1), the partial state A_ij = (O_ij, L_ij): O normalised
// over the visible keys of the item, L = natural-log LSE of the masked scaled
// scores.  The key tiles stream through the online recurrence of "上下文并行"
// 02 ONE ROW (running max m, denominator l, accumulator a in TMEM).
//
// Persistent kernel, one CTA per SM, 192 threads in three roles:
//   warp 0       TMA producer: Q tile (once per item), K and V tiles (2-stage
//                rings), 128-byte-swizzled boxes of 64 x 128 bf16;
//   warp 1       tcgen05.mma issuer (one lane): S = Q K^T into one of two
//                TMEM S buffers (M=128, N=128, K=16 per instruction, fp32),
//                then O += P V with V read MN-major; owns the TMEM allocation;
//   warps 2..5   softmax: one query row per thread (TMEM lane), masking by
//                original position, exp2 on the MUFU, P written to shared
//                memory as bf16 in the MMA's swizzled K-major layout, lazy
//                rescale of O in TMEM (only when the row max grows by more than
//                2^8), epilogue O / l and L = (m + log2 l) ln 2.
// Work items are taken in a static round-robin over (batch, head, item) with
// items sorted heaviest first.  Every mbarrier wait is bounded; on timeout the
// block raises the device error word, drains its copies and frees TMEM.
#include <cuda_bf16.h>

#include "internal.h"
#include "tc_util.cuh"
#include "tmap.h"

namespace cpattn {

namespace {

// Opt-in timeline trace (build with -DCPATTN_TRACE): block 0 records
// (event, tile, clock64) triples for the first kTraceMax events.
#ifdef CPATTN_TRACE
constexpr int kTraceTiles = 4096, kTraceEvents = 8;
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

constexpr int kThreads = 320;
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile = 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 128 x 64 swizzled box
constexpr int kOffQ = 0;
constexpr int kStages = 3;                         // K and V ring depth
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffX = kOffV + kStages * kTileBytes;  // row max / sum exchange, 2 KB
constexpr int kOffBar = kOffX + 2048;
constexpr int kSmemBytes = kOffBar + 256;

// barrier slots (8 bytes each)
enum {
  B_QFULL = 0, B_QEMPTY, B_KFULL0, B_KEMPTY0 = B_KFULL0 + kStages, B_VFULL0 = B_KEMPTY0 + kStages,
  B_VEMPTY0 = B_VFULL0 + kStages, B_SFULL0 = B_VEMPTY0 + kStages, B_SFULL1, B_SFULL2, B_PCONS0, B_PCONS1, B_PCONS2, B_PFULL0, B_PFULL1, B_PFULL2,
  B_PVDONE, B_ODONE, B_XCH0, B_XCH1, B_XCH2, B_XCH3, B_DRAIN, B_COUNT
};

constexpr uint32_t kIdescS = tc::idesc_bf16(128, 128, /*b_mn_major=*/0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, /*b_mn_major=*/1);

struct Params {
  CUtensorMap tmq, tmk, tmv;
  FwdArgs a;
  int* err;
  float scale_log2;
  int64_t total_work;
};

struct Item {
  int32_t row0, pos0, len, out_row0;
  int32_t n_seg;
  Seg seg[2];
  int32_t eff[2];
  int32_t ntile[2];
  int32_t n;  // key tiles
};

__device__ __forceinline__ Item load_item(const FwdArgs& a, int idx) {
  Item it;
  if (a.items) {
    const TileItem t = a.items[idx];
    it.row0 = t.row0;
    it.pos0 = t.pos0;
    it.len = t.len;
    it.out_row0 = t.out_row0;
    it.n_seg = t.seg_count < 2 ? t.seg_count : 2;
    for (int s = 0; s < 2; ++s) it.seg[s] = s < it.n_seg ? a.segs[t.seg_begin + s] : Seg{0, 0, 0, 0};
  } else {
    it.row0 = a.edge.q_row0 + idx * kTile;
    it.pos0 = a.edge.q_pos0 + idx * kTile;
    it.len = min(kTile, a.edge.q_len - idx * kTile);
    it.out_row0 = idx * kTile;
    it.n_seg = 1;
    it.seg[0] = Seg{a.edge.kv_row0, a.edge.kv_pos0, a.edge.kv_len, 0};
    it.seg[1] = Seg{0, 0, 0, 0};
  }
  const int qlast = it.pos0 + it.len - 1;
  it.n = 0;
  for (int s = 0; s < 2; ++s) {
    int e = s < it.n_seg ? it.seg[s].len : 0;
    if (a.causal) e = min(e, qlast - it.seg[s].pos0 + 1);
    e = max(e, 0);
    it.eff[s] = e;
    it.ntile[s] = (e + kTile - 1) / kTile;
    it.n += it.ntile[s];
  }
  return it;
}

// Key tile t of an item: segment and offset.
__device__ __forceinline__ void tile_of(const Item& it, int t, int& s, int& kt) {
  s = t < it.ntile[0] ? 0 : 1;
  kt = (s == 0 ? t : t - it.ntile[0]) * kTile;
}

__device__ __forceinline__ void decode_work(const Params& p, int64_t w, int& item, int& b, int& h) {
  const int64_t bh = w / p.a.n_items;
  item = int(w - bh * p.a.n_items);
  b = int(bh / p.a.H);
  h = int(bh - int64_t(b) * p.a.H);
}

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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FwdArgs& a = p.a;

  if (threadIdx.x == 0) {
    tc::mbar_init(bar(B_QFULL), 1);
    tc::mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar(B_KFULL0 + s), 1);
      tc::mbar_init(bar(B_KEMPTY0 + s), 1);
      tc::mbar_init(bar(B_VFULL0 + s), 1);
      tc::mbar_init(bar(B_VEMPTY0 + s), 1);
    }
    for (int s = 0; s < 3; ++s) {
      tc::mbar_init(bar(B_SFULL0 + s), 1);
      tc::mbar_init(bar(B_PCONS0 + s), 1);
    }
    for (int s = 0; s < 3; ++s) tc::mbar_init(bar(B_PFULL0 + s), 256);  // one per S/P buffer
    tc::mbar_init(bar(B_PVDONE), 1);
    tc::mbar_init(bar(B_ODONE), 1);
    for (int q = 0; q < 4; ++q) tc::mbar_init(bar(B_XCH0 + q), 64);  // the two warps of a quarter
    tc::mbar_init(bar(B_DRAIN), 1);
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
  // three S buffers (P overwrites the S it came from) and the O accumulator
  const uint32_t tS0 = tmem, tO = tmem + 384;

  const int64_t first = blockIdx.x, stride = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tc::prefetch_tmap(&p.tmq);
      tc::prefetch_tmap(&p.tmk);
      tc::prefetch_tmap(&p.tmv);
      uint32_t g = 0, qi = 0;
      bool ok = true;
      uint32_t armed_q = 0, armed_k[kStages] = {}, armed_v[kStages] = {};  // uses armed so far
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        const int g_kv = h / (a.H / a.Hkv);
        const int64_t rbase = int64_t(b) * a.seqlen;
        ok = tc::mbar_wait(bar(B_QEMPTY), (qi & 1) ^ 1, abort_flag, p.err);
        if (!ok) break;
        tc::mbar_arrive_expect_tx(bar(B_QFULL), kTileBytes);
        tc::tma_load_3d(sQ, &p.tmq, bar(B_QFULL), 0, h, int(rbase + it.row0));
        tc::tma_load_3d(sQ + kHalfBytes, &p.tmq, bar(B_QFULL), 64, h, int(rbase + it.row0));
        ++armed_q;
        ++qi;
        for (int t = 0; t < it.n && ok; ++t, ++g) {
          int s, kt;
          tile_of(it, t, s, kt);
          const int row = int(rbase + it.seg[s].row0 + kt);
          const uint32_t st = g % kStages, ph = (g / kStages) & 1;
          ok = tc::mbar_wait(bar(B_KEMPTY0 + st), ph ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(bar(B_KFULL0 + st), kTileBytes);
          tc::tma_load_3d(sK + st * kTileBytes, &p.tmk, bar(B_KFULL0 + st), 0, g_kv, row);
          tc::tma_load_3d(sK + st * kTileBytes + kHalfBytes, &p.tmk, bar(B_KFULL0 + st), 64, g_kv, row);
          ++armed_k[st];
          FWD_TRACE(1, g);
          ok = tc::mbar_wait(bar(B_VEMPTY0 + st), ph ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(bar(B_VFULL0 + st), kTileBytes);
          tc::tma_load_3d(sV + st * kTileBytes, &p.tmv, bar(B_VFULL0 + st), 0, g_kv, row);
          tc::tma_load_3d(sV + st * kTileBytes + kHalfBytes, &p.tmv, bar(B_VFULL0 + st), 64, g_kv, row);
          ++armed_v[st];
        }
      }
      // Drain: every copy this thread started has landed before the block exits.
      volatile int never = 0;
      if (armed_q) tc::mbar_wait(bar(B_QFULL), (armed_q - 1) & 1, &never, nullptr);
      for (int s = 0; s < kStages; ++s) {
        if (armed_k[s]) tc::mbar_wait(bar(B_KFULL0 + s), (armed_k[s] - 1) & 1, &never, nullptr);
        if (armed_v[s]) tc::mbar_wait(bar(B_VFULL0 + s), (armed_v[s] - 1) & 1, &never, nullptr);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint64_t qd = tc::kmajor_desc(sQ);
      uint32_t g = 0, qi = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t gi, bool first_tile) -> bool {
        if (!tc::mbar_wait(bar(B_PFULL0 + gi % 3), (gi / 3) & 1, abort_flag, p.err)) return false;
        if (!tc::mbar_wait(bar(B_VFULL0 + gi % kStages), (gi / kStages) & 1, abort_flag, p.err)) return false;
        tc::fence_after_sync();
        const uint64_t vd = tc::mnmajor_desc(sV + (gi % kStages) * kTileBytes);
        const uint32_t pcol = tS0 + (gi % 3) * 128;
        const uint32_t acc0 = first_tile ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // P (bf16, TMEM, over S) x V (MN-major smem)
          tc::mma_ts(tO, pcol + (kk >> 2) * 64 + (kk & 3) * 8, tc::mnmajor_step(vd, kk), kIdescPV,
                     kk == 0 ? acc0 : 1u);
        tc::mma_commit(bar(B_VEMPTY0 + gi % kStages));
        tc::mma_commit(bar(B_PCONS0 + gi % 3));  // this S/P buffer may be overwritten
        tc::mma_commit(bar(B_PVDONE));
        FWD_TRACE(3, gi);
        return true;
      };
      for (int64_t w = first; w < p.total_work && ok; w += stride) {
        int idx, b, h;
        decode_work(p, w, idx, b, h);
        const Item it = load_item(a, idx);
        if (it.n == 0) continue;
        ok = tc::mbar_wait(bar(B_QFULL), qi & 1, abort_flag, p.err);
        ++qi;
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t g0 = g;
        for (int t = 0; t < it.n && ok; ++t, ++g) {
          const uint32_t st = g % kStages;
          ok = tc::mbar_wait(bar(B_KFULL0 + st), (g / kStages) & 1, abort_flag, p.err);
          // the S buffer's previous P must have been read by its PV
          if (ok) ok = tc::mbar_wait(bar(B_PCONS0 + g % 3), ((g / 3) & 1) ^ 1, abort_flag, p.err);
          if (!ok) break;
          tc::fence_after_sync();
          const uint64_t kd = tc::kmajor_desc(sK + st * kTileBytes);
          const uint32_t scol = tS0 + (g % 3) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_ss(scol, tc::kmajor_step(qd, kk), tc::kmajor_step(kd, kk), kIdescS, kk > 0 ? 1u : 0u);
          tc::mma_commit(bar(B_KEMPTY0 + st));
          tc::mma_commit(bar(B_SFULL0 + g % 3));
          FWD_TRACE(2, g);
          if (t == it.n - 1) tc::mma_commit(bar(B_QEMPTY));
          if (t >= 1) ok = issue_pv(g - 1, t - 1 == 0);
        }
        if (ok) ok = issue_pv(g - 1, it.n == 1);
        if (ok) tc::mma_commit(bar(B_ODONE));  // O of this item is final
        (void)g0;
      }
      // Drain: all MMAs issued by this thread are complete before TMEM is freed.
      volatile int never = 0;
      tc::mma_commit(bar(B_DRAIN));
      tc::mbar_wait(bar(B_DRAIN), 0, &never, nullptr);
    }
  } else {
    // ----------------------------------------------------- softmax warps --
    // Eight warps, two per TMEM lane quarter: warp w serves query rows
    // 32 (w % 4) .. +31 and key / output columns 64 h .. 64 h + 63 with
    // h = (w - 2) / 4.  The two warps of a quarter exchange their partial row
    // maxima (and, at the end, row sums) through shared memory.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;            // query row in the tile = TMEM lane
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const int xbar = B_XCH0 + quarter;              // exchange barrier of the two warps
    float* xbuf = reinterpret_cast<float*>(smem + kOffX);  // [exchange parity][half][row]
    const float sl2 = p.scale_log2;
    uint32_t g = 0, oi = 0, xc = 0;
    bool ok = true;
    for (int64_t w = first; w < p.total_work && ok; w += stride) {
      int idx, b, h;
      decode_work(p, w, idx, b, h);
      const Item it = load_item(a, idx);
      const int qpos = it.pos0 + row;
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < it.n && ok; ++t, ++g) {
        int s, kt;
        tile_of(it, t, s, kt);
        const uint32_t sb = g % 3;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_SFULL0 + sb), (g / 3) & 1, abort_flag, p.err));
        if (threadIdx.x == 64) FWD_TRACE(4, g);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t taddr = tS0 + sb * 128 + lane_off + half * 64;
        // visible keys of this row in this tile: j < limit
        const int kpos0 = it.seg[s].pos0 + kt;
        int limit = min(kTile, it.eff[s] - kt);
        if (a.causal) limit = min(limit, qpos - kpos0 + 1);
        limit -= half * 64;  // in this warp's column range
        // this warp's 64 scores of the row, one TMEM round trip; row max of the
        // scaled, masked scores (own half, then the pair's)
        uint32_t sr[64];
        tc::tmem_ld32(taddr, sr);
        tc::tmem_ld32(taddr + 32, sr + 32);
        tc::tmem_wait_ld();
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) mx = fmaxf(mx, j < limit ? __uint_as_float(sr[j]) : -INFINITY);
        mx *= sl2;
        xbuf[((xc & 1) * 2 + half) * 128 + row] = mx;
        tc::mbar_arrive(bar(xbar));
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(xbar), xc & 1, abort_flag, p.err));
        if (!ok) break;
        mx = fmaxf(mx, xbuf[((xc & 1) * 2 + (half ^ 1)) * 128 + row]);
        if (threadIdx.x == 64) FWD_TRACE(5, g);
        ++xc;
        const float m_new = fmaxf(m, mx);
        const bool grow = m_new > m + 8.0f;  // also true when m is -inf and m_new finite
        float corr = 1.f;
        if (grow) {
          corr = (m == -INFINITY) ? 0.f : tc::ex2(m - m_new);
          m = m_new;
          l *= corr;
        }
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
          // O may only be rescaled once PV of the previous tile is done
          ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_PVDONE), (g - 1) & 1, abort_flag, p.err));
          if (!ok) break;
          tc::fence_after_sync();
          uint32_t orr[64];
          tc::tmem_ld32(tO + lane_off + half * 64, orr);
          tc::tmem_ld32(tO + lane_off + half * 64 + 32, orr + 32);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 64; ++j) orr[j] = __float_as_uint(__uint_as_float(orr[j]) * corr);
          tc::tmem_st32(tO + lane_off + half * 64, orr);
          tc::tmem_st32(tO + lane_off + half * 64 + 32, orr + 32);
          tc::tmem_wait_st();
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        // P = exp2(x - m) as bf16 pairs over the consumed S columns of this
        // half (keys 2c, 2c+1 -> column c of the half)
        float lsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j0 = cc * 32 + 2 * e;
            const float x0 = j0 < limit ? fmaf(__uint_as_float(sr[j0]), sl2, -mu) : -INFINITY;
            const float x1 = j0 + 1 < limit ? fmaf(__uint_as_float(sr[j0 + 1]), sl2, -mu) : -INFINITY;
            const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
            lsum += p0 + p1;
            pk[e] = tc::pack_bf16x2(p0, p1);
          }
          tc::tmem_st16(taddr + cc * 16, pk);
        }
        l += lsum;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(bar(B_PFULL0 + g % 3));
        if (threadIdx.x == 64) FWD_TRACE(6, g);
      }
      if (!ok) break;
      // ------------------------------------------------------ epilogue --
      if (it.n > 0) {
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_ODONE), oi & 1, abort_flag, p.err));
        ++oi;
        if (!ok) break;
        tc::fence_after_sync();
      }
      xbuf[((xc & 1) * 2 + half) * 128 + row] = l;
      tc::mbar_arrive(bar(xbar));
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(xbar), xc & 1, abort_flag, p.err));
      if (!ok) break;
      l += xbuf[((xc & 1) * 2 + (half ^ 1)) * 128 + row];
      ++xc;
      {
        const bool store = row < it.len;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t prow_i = (int64_t(b) * a.part_rows + it.out_row0 + row) * a.H + h;
        float4* dst = reinterpret_cast<float4*>(a.o_part + prow_i * 128 + half * 64);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t orr[32];
          if (it.n > 0) {
            tc::tmem_ld32(tO + lane_off + half * 64 + cc * 32, orr);
            tc::tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) orr[j] = 0u;
          }
          if (store) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[cc * 8 + j] = make_float4(__uint_as_float(orr[4 * j]) * inv, __uint_as_float(orr[4 * j + 1]) * inv,
                                            __uint_as_float(orr[4 * j + 2]) * inv, __uint_as_float(orr[4 * j + 3]) * inv);
          }
        }
        tc::fence_before_sync();
        if (store && half == 0) a.lse_part[prow_i] = l > 0.f ? (m + tc::lg2(l)) * 0.69314718055994531f : -INFINITY;
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

bool fwd_tc_supported(const FwdArgs& a) {
  return a.dtype == CP_BF16 && a.d == 128 && tmap_encoder() != nullptr;
}

#ifdef CPATTN_TRACE
extern "C" int cp_fwd_trace_dump(unsigned long long* out, int max_events) {
  cudaDeviceSynchronize();
  const int n = max_events < kTraceEvents * kTraceTiles ? max_events : kTraceEvents * kTraceTiles;
  cudaMemcpyFromSymbol(out, g_fwd_trace, sizeof(unsigned long long) * n);
  return n;
}
#endif

cp_status launch_fwd_tc(const FwdArgs& a, cudaStream_t s) {
  if (a.n_items == 0) return CP_OK;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return CP_ERR_CUDA;
    attr_set[dev] = true;
  }
  Params p;
  const int64_t rows = int64_t(a.batch) * a.seqlen;
  if (!make_tmap_rows(&p.tmq, a.q, rows, a.H, 128, 128) ||
      !make_tmap_rows(&p.tmk, a.k, rows, a.Hkv, 128, 128) ||
      !make_tmap_rows(&p.tmv, a.v, rows, a.Hkv, 128, 128))
    return CP_ERR_CUDA;
  p.a = a;
  p.err = device_error_ptr();
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.total_work = int64_t(a.n_items) * a.batch * a.H;
  const int64_t grid = p.total_work < num_sms() ? p.total_work : num_sms();
  fwd_tc_kernel<<<unsigned(grid), kThreads, kSmemBytes, s>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
