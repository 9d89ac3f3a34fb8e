// LSE merge of partial states ("Context Parallelism (CP)" §2.2):
//   L_i = log sum_j exp L_ij,   O_i = sum_j exp(L_ij - L_i) O_ij.
// One warp per (row, head): lane j < n_parts holds L_ij, the max and the sum
// are warp shuffles, the weights exp(L_ij - L_i) are shuffled from lane j, and
// each partial's O row (head_dim floats) is one coalesced vector load per
// lane, four partial rows in flight at a time.  Memory bound: n_parts *
// (4 d + 4) bytes read and d * elem + 4 bytes written per (row, head).
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "internal.h"

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

template <typename TO, int D>
__global__ void __launch_bounds__(256) merge_kernel(MergeArgs a) {
  constexpr int kPer = D / 32;  // floats per lane
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int H = a.H;
  const int64_t total = a.merge_rows * H;
  const int b = blockIdx.y;
  const float* o_base = a.o_part + int64_t(b) * a.part_rows * H * D;
  const float* l_base = a.lse_part + int64_t(b) * a.part_rows * H;
  for (int64_t w = warp; w < total; w += n_warps) {
    const int32_t m = int32_t(w / H);
    const int h = int(w - int64_t(m) * H);
    const MergeSeg sg = a.segs ? *find_seg(a.segs, a.n_segs, m) : a.dense;
    const int32_t i = m - sg.merge_row0;
    const int np = sg.n_parts;
    auto prow_of = [&](int e) { return int64_t(sg.part_row0) + int64_t(e) * sg.part_stride + i; };
    // L of every partial of this row (lane e holds L_e): max, then the
    // log-sum-exp
    float l_lane = -INFINITY, mx = -INFINITY;
    for (int e = lane; e < np; e += 32) {
      const float le = l_base[prow_of(e) * H + h];
      if (e == lane) l_lane = le;
      mx = fmaxf(mx, le);
    }
    mx = warp_max(mx);
    const float base = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
    for (int e = lane; e < np; e += 32) sum += expf((e == lane ? l_lane : l_base[prow_of(e) * H + h]) - base);
    sum = warp_sum(sum);
    const float lse = (mx == -INFINITY) ? -INFINITY : base + logf(sum);
    float acc[kPer];
#pragma unroll
    for (int t = 0; t < kPer; ++t) acc[t] = 0.f;
    if (mx != -INFINITY) {
      if (np <= 32) {
        // weights exp(L_e - L) from lane e; four partial rows in flight per step
        const float w_lane = lane < np ? expf(l_lane - lse) : 0.f;  // 0 for -inf partials
        int e = 0;
        for (; e + 4 <= np; e += 4) {
          float x[4][kPer];
#pragma unroll
          for (int j = 0; j < 4; ++j) load_vec<float, kPer>(o_base + (prow_of(e + j) * H + h) * D + lane * kPer, x[j]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float wgt = __shfl_sync(0xffffffffu, w_lane, e + j);
#pragma unroll
            for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[j][t], acc[t]);
          }
        }
        for (; e < np; ++e) {
          float x[kPer];
          load_vec<float, kPer>(o_base + (prow_of(e) * H + h) * D + lane * kPer, x);
          const float wgt = __shfl_sync(0xffffffffu, w_lane, e);
#pragma unroll
          for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[t], acc[t]);
        }
      } else {
        for (int e = 0; e < np; ++e) {
          const int64_t prow = prow_of(e);
          const float wgt = expf(l_base[prow * H + h] - lse);  // 0 for -inf partials
          float x[kPer];
          load_vec<float, kPer>(o_base + (prow * H + h) * D + lane * kPer, x);
#pragma unroll
          for (int t = 0; t < kPer; ++t) acc[t] = fmaf(wgt, x[t], acc[t]);
        }
      }
    }
    const int64_t orow = int64_t(b) * a.out_rows + sg.out_row0 + i;
    store_vec<TO, kPer>(static_cast<TO*>(a.o_out) + (orow * H + h) * D + lane * kPer, acc);
    if (a.lse_out && lane == 0) a.lse_out[orow * H + h] = lse;
  }
}

}  // namespace

cp_status launch_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t total = a.merge_rows * a.H;
  if (total == 0) return CP_OK;
  int64_t blocks = (total + 7) / 8;
  const int64_t cap = 152 * 16;
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
