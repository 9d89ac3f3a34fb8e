// LSE merge of partial states ("Context Parallelism (CP)" §2.2):
//   L_i = log sum_j exp L_ij,   O_i = sum_j exp(L_ij - L_i) O_ij.
// One warp per merged row and all its heads; each partial's O row (head_dim
// floats) is one coalesced vector load per lane.  Memory bound: n_parts *
// (4 d + 4) bytes read and d * elem + 4 bytes written per (row, head).
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "internal.h"
#include "tmap.h"

namespace cpattn {

namespace {

__device__ __forceinline__ const MergeSeg* find_seg(const MergeSeg* segs, int n, int32_t m) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].merge_row0 <= m) lo = mid; else hi = mid - 1;
  }
  return segs + lo;
}

// Merge of one (row, head).  Up to kFew partials: every lane reads the L
// values itself (broadcast loads) and forms the weights, no shuffles; the O
// rows are requested before the L arithmetic.  More partials: lane e holds
// L_e, warp shuffles give the max, the sum and the weights, four O rows in
// flight at a time.
constexpr int kFew = 4;

template <typename TO, int D>
__device__ __forceinline__ void merge_row_head(const float* __restrict__ o_base, const float* __restrict__ l_base,
                                               int64_t prow0, int64_t pstride, int np, int H, int h, int lane,
                                               TO* __restrict__ o_dst, float* __restrict__ lse_dst) {
  constexpr int kPer = D / 32;
  auto orow = [&](int e) { return o_base + ((prow0 + int64_t(e) * pstride) * H + h) * D + lane * kPer; };
  auto lval = [&](int e) { return l_base[(prow0 + int64_t(e) * pstride) * H + h]; };
  float acc[kPer];
#pragma unroll
  for (int t = 0; t < kPer; ++t) acc[t] = 0.f;
  float lse;
  if (np <= kFew) {
    float x[kFew][kPer], L[kFew];
#pragma unroll
    for (int j = 0; j < kFew; ++j) {
      if (j < np) {
        load_vec<float, kPer>(orow(j), x[j]);
        L[j] = lval(j);
      } else {
#pragma unroll
        for (int t = 0; t < kPer; ++t) x[j][t] = 0.f;
        L[j] = -INFINITY;
      }
    }
    float mx = L[0];
#pragma unroll
    for (int j = 1; j < kFew; ++j) mx = fmaxf(mx, L[j]);
    if (mx == -INFINITY) {
      lse = -INFINITY;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kFew; ++j) sum += expf(L[j] - mx);  // 0 for -inf partials
      lse = mx + logf(sum);
#pragma unroll
      for (int j = 0; j < kFew; ++j) {
        const float wgt = expf(L[j] - lse);
#pragma unroll
        for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[j][t], acc[t]);
      }
    }
  } else {
    float l_lane = -INFINITY, mx = -INFINITY;
    for (int e = lane; e < np; e += 32) {
      const float le = lval(e);
      if (e == lane) l_lane = le;
      mx = fmaxf(mx, le);
    }
    mx = warp_max(mx);
    const float base = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
    for (int e = lane; e < np; e += 32) sum += expf((e == lane ? l_lane : lval(e)) - base);
    sum = warp_sum(sum);
    lse = (mx == -INFINITY) ? -INFINITY : base + logf(sum);
    if (mx != -INFINITY) {
      if (np <= 32) {
        const float w_lane = lane < np ? expf(l_lane - lse) : 0.f;  // 0 for -inf partials
        int e = 0;
        for (; e + 4 <= np; e += 4) {
          float x[4][kPer];
#pragma unroll
          for (int j = 0; j < 4; ++j) load_vec<float, kPer>(orow(e + j), x[j]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float wgt = __shfl_sync(0xffffffffu, w_lane, e + j);
#pragma unroll
            for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[j][t], acc[t]);
          }
        }
        for (; e < np; ++e) {
          float x[kPer];
          load_vec<float, kPer>(orow(e), x);
          const float wgt = __shfl_sync(0xffffffffu, w_lane, e);
#pragma unroll
          for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[t], acc[t]);
        }
      } else {
        for (int e = 0; e < np; ++e) {
          const float wgt = expf(lval(e) - lse);  // 0 for -inf partials
          float x[kPer];
          load_vec<float, kPer>(orow(e), x);
#pragma unroll
          for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[t], acc[t]);
        }
      }
    }
  }
  store_vec<TO, kPer>(o_dst + lane * kPer, acc);
  if (lse_dst && lane == 0) *lse_dst = lse;
}

// One warp per merged row, all heads of it (the segment lookup and the row
// arithmetic once per row), two heads in flight.
template <typename TO, int D>
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int H = a.H;
  const int b = blockIdx.y;
  const float* o_base = a.o_part + int64_t(b) * a.part_rows * H * D;
  const float* l_base = a.lse_part + int64_t(b) * a.part_rows * H;
  for (int64_t m = warp; m < a.merge_rows; m += n_warps) {
    const MergeSeg sg = a.segs ? *find_seg(a.segs, a.n_segs, int32_t(m)) : a.dense;
    const int32_t i = int32_t(m) - sg.merge_row0;
    const int64_t prow0 = int64_t(sg.part_row0) + i;
    const int64_t orow = int64_t(b) * a.out_rows + sg.out_row0 + i;
    TO* o_dst = static_cast<TO*>(a.o_out) + orow * H * D;
    float* l_dst = a.lse_out ? a.lse_out + orow * H : nullptr;
#pragma unroll 2
    for (int h = 0; h < H; ++h)
      merge_row_head<TO, D>(o_base, l_base, prow0, sg.part_stride, sg.n_parts, H, h, lane, o_dst + int64_t(h) * D,
                            l_dst ? l_dst + h : nullptr);
  }
}

}  // namespace

cp_status launch_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t total = a.merge_rows;
  if (total == 0 || a.H == 0) return CP_OK;
  int64_t blocks = (total + 7) / 8;  // 8 warps (rows) per block
  const int64_t cap = int64_t(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  const dim3 grid(unsigned(blocks), unsigned(a.batch));
  if (a.out_dtype == CP_BF16) {
    if (a.d == 128) merge_kernel<__nv_bfloat16, 128><<<grid, 256, 0, s>>>(a);
    else merge_kernel<__nv_bfloat16, 64><<<grid, 256, 0, s>>>(a);
  } else {
    if (a.d == 128) merge_kernel<float, 128><<<grid, 256, 0, s>>>(a);
    else merge_kernel<float, 64><<<grid, 256, 0, s>>>(a);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
