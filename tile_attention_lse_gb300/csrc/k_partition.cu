// Partition index kernel and token gather ("04 · Megatron-LM 实现" §1.1:
// view as 2*cp chunks, rank r keeps chunks r and 2cp-1-r, then index_select;
// §1.2: the same inside every packed sub-sequence; "Context Parallelism (CP)"
// §4).
#include <cuda_bf16.h>

#include <cmath>

#include "device_util.cuh"
#include "internal.h"
#include "tmap.h"

namespace cpattn {

// One thread per rank-local slot g = r * (L / cp) + t.
//  BSHD (cu == nullptr): c = L / (2cp); slot t < c -> chunk r, else chunk 2cp-1-r.
//  THD: the rank's local stream is sub-sequence major; sub-sequence k occupies
//  local slots [cu[k] / cp, cu[k+1] / cp), front chunk then mirrored chunk.
//  striped: the same slots, the u-th slot of sub-sequence k on rank r is token
//  start_k + r + cp * u ("Sequence Parallelism + Ring Attention" §5).
__global__ void __launch_bounds__(256) partition_kernel(int32_t cp, int64_t L,
                                                        const int32_t* __restrict__ cu,
                                                        int32_t n_seqs, int32_t* __restrict__ idx,
                                                        int32_t* __restrict__ local_cu, int striped) {
  const int64_t per_rank = L / cp;
  const int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (local_cu && g <= n_seqs) local_cu[g] = cu[g] / cp;
  if (g >= L) return;
  const int r = int(g / per_rank);
  const int64_t t = g - int64_t(r) * per_rank;
  int64_t start = 0, c = L / (2 * cp), off = t;
  if (cu) {
    // largest k with cu[k] / cp <= t  (lengths may be zero: take the last such k
    // whose sub-sequence is non-empty, i.e. cu[k+1] / cp > t)
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (int64_t(cu[mid]) / cp <= t) lo = mid; else hi = mid - 1;
    }
    start = cu[lo];
    c = (int64_t(cu[lo + 1]) - cu[lo]) / (2 * cp);
    off = t - start / cp;
  }
  if (striped) {
    idx[g] = int32_t(start + r + int64_t(cp) * off);
    return;
  }
  const int64_t chunk = off < c ? r : 2 * cp - 1 - r;
  const int64_t within = off < c ? off : off - c;
  idx[g] = int32_t(start + chunk * c + within);
}

cp_status launch_partition(int32_t cp, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                           int32_t* idx, int32_t* local_cu, int striped, cudaStream_t s) {
  const int64_t n = seqlen > n_seqs + 1 ? seqlen : n_seqs + 1;
  const unsigned blocks = unsigned((n + 255) / 256);
  partition_kernel<<<blocks, 256, 0, s>>>(cp, seqlen, cu_dev, n_seqs, idx, local_cu, striped);
  return cuda_status(cudaGetLastError());
}

// Hybrid CP layout ("04 · Megatron-LM 实现" §7 and §1.1: each sub-sequence k
// zigzag-split with cp = seq_cp[k] over ranks seq_rank0[k] ..).  Rank r's
// stream holds, sub-sequence by sub-sequence, its slices of the
// sub-sequences whose group contains it; the streams follow each other in
// rank order.
//  Pass 1, one block per rank: where each slice of rank r starts
//  (local_cu[r][k]) and where the stream ends (local_cu[r][n]).
//  Pass 2, one thread per original token: its rank, slice and slot.
__device__ __forceinline__ int64_t hybrid_slice(const int32_t* cu, const int32_t* gcp, const int32_t* g0, int k,
                                                int r) {
  const int g = gcp[k], o = r - g0[k];
  return (g > 0 && o >= 0 && o < g) ? int64_t(cu[k + 1] - cu[k]) / g : 0;
}

__global__ void __launch_bounds__(256) hybrid_slices_kernel(const int32_t* __restrict__ cu,
                                                            const int32_t* __restrict__ gcp,
                                                            const int32_t* __restrict__ g0, int32_t n_seqs,
                                                            int32_t* __restrict__ local_cu) {
  __shared__ int64_t warp_sum[8];
  __shared__ int64_t carry;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // start of rank r's stream: the slices of every lower rank
  int64_t before = 0;
  for (int k = tid; k < n_seqs; k += 256) {
    const int g = gcp[k];
    const int lower = min(max(r - g0[k], 0), g);
    if (g > 0) before += int64_t(cu[k + 1] - cu[k]) / g * lower;
  }
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) warp_sum[warp] = before;
  __syncthreads();
  if (tid == 0) {
    int64_t x = 0;
    for (int w = 0; w < 8; ++w) x += warp_sum[w];
    carry = x;
  }
  __syncthreads();
  // exclusive scan of this rank's slice lengths, 256 sub-sequences at a time
  int32_t* out = local_cu + int64_t(r) * (n_seqs + 1);
  for (int k0 = 0; k0 <= n_seqs; k0 += 256) {
    const int k = k0 + tid;
    const int64_t v = k < n_seqs ? hybrid_slice(cu, gcp, g0, k, r) : 0;
    int64_t incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int64_t base = carry;
    for (int w = 0; w < warp; ++w) base += warp_sum[w];
    if (k <= n_seqs) out[k] = int32_t(base + incl - v);
    __syncthreads();
    if (tid == 255) carry = base + incl;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) hybrid_index_kernel(int64_t T, int32_t n_ranks, const int32_t* __restrict__ cu,
                                                           const int32_t* __restrict__ gcp,
                                                           const int32_t* __restrict__ g0, int32_t n_seqs,
                                                           const int32_t* __restrict__ local_cu,
                                                           int32_t* __restrict__ idx) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= T) return;
  // the sub-sequence holding t: the last k with cu[k] <= t (empty ones end
  // where the next starts, so the last such k is non-empty)
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int k = lo, g = gcp[k];
  const int64_t p = t - cu[k], c = g > 0 ? int64_t(cu[k + 1] - cu[k]) / (2 * g) : 0;
  if (c <= 0) return;  // device copies disagree with the validated host arrays
  const int64_t a = p / c;
  const int o = int(a < g ? a : 2 * g - 1 - a);
  const int64_t within = (a < g ? 0 : c) + (p - a * c);
  const int r = g0[k] + o;
  if (r < 0 || r >= n_ranks) return;
  const int64_t slot = local_cu[int64_t(r) * (n_seqs + 1) + k] + within;
  if (slot >= 0 && slot < T) idx[slot] = int32_t(t);
}

cp_status launch_partition_hybrid(int32_t cp, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                                  const int32_t* gcp_dev, const int32_t* g0_dev, int32_t* idx, int32_t* local_cu,
                                  cudaStream_t s) {
  hybrid_slices_kernel<<<unsigned(cp), 256, 0, s>>>(cu_dev, gcp_dev, g0_dev, n_seqs, local_cu);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || seqlen == 0) return cuda_status(e);
  hybrid_index_kernel<<<unsigned((seqlen + 255) / 256), 256, 0, s>>>(seqlen, cp, cu_dev, gcp_dev, g0_dev, n_seqs,
                                                                     local_cu, idx);
  return cuda_status(cudaGetLastError());
}

// Sub-sequence and in-sequence position of the token at every rank-local
// slot: one thread per slot, a binary search in cu for packed input.
__global__ void __launch_bounds__(256) token_seq_pos_kernel(const int32_t* __restrict__ idx, int64_t T,
                                                            const int32_t* __restrict__ cu, int32_t n_seqs,
                                                            int32_t* __restrict__ seq_pos) {
  const int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= T) return;
  const int32_t t = idx[g];
  int k = 0, start = 0;
  if (cu) {
    // the last k with cu[k] <= t (empty sub-sequences end where the next starts)
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    k = lo;
    start = cu[k];
  }
  seq_pos[2 * g] = k;
  seq_pos[2 * g + 1] = t - start;
}

cp_status launch_token_seq_pos(const int32_t* idx, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                               int32_t* seq_pos, cudaStream_t s) {
  token_seq_pos_kernel<<<unsigned((seqlen + 255) / 256), 256, 0, s>>>(idx, seqlen, cu_dev, n_seqs, seq_pos);
  return cuda_status(cudaGetLastError());
}

// Row gather with 16-byte vectors: one warp-strided loop per row.  A row is
// heads * head_dim elements (row_bytes, a multiple of 16).
__global__ void __launch_bounds__(256) permute_kernel(const int32_t* __restrict__ idx,
                                                      int64_t seqlen, int64_t rows_total,
                                                      int64_t row_vecs, const uint4* __restrict__ src,
                                                      uint4* __restrict__ dst, int inverse) {
  const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows_total;
       row += warps) {
    const int64_t b = row / seqlen;
    const int64_t t = row - b * seqlen;
    const int64_t other = b * seqlen + idx[t];
    const int64_t s_row = inverse ? row : other;
    const int64_t d_row = inverse ? other : row;
    const uint4* ps = src + s_row * row_vecs;
    uint4* pd = dst + d_row * row_vecs;
    for (int64_t v = lane; v < row_vecs; v += 32) pd[v] = ps[v];
  }
}

cp_status launch_permute(const int32_t* idx, int32_t batch, int64_t seqlen, int64_t row_bytes,
                         const void* src, void* dst, int inverse, cudaStream_t s) {
  if (row_bytes % 16) return CP_ERR_UNSUPPORTED;
  const int64_t rows = int64_t(batch) * seqlen;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > int64_t(num_sms()) * 16) blocks = int64_t(num_sms()) * 16;
  permute_kernel<<<unsigned(blocks), 256, 0, s>>>(idx, seqlen, rows, row_bytes / 16,
                                                  static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst), inverse);
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Token gather with rotary position embedding ("04 · Megatron-LM 实现" §5: the
// positions are split by the same zigzag as the tokens).  One warp per token
// row and all its heads.  pos = the token's position in its sequence
// (BSHD: the original index; THD: the index minus its sub-sequence start).
// For pair i < D/2 the angle is pos * inv_freq[i], formed and reduced to
// [-pi, pi] in float64 (an float32 product at pos ~1e5 would be off by ~1e-2
// rad), then sin/cos in float32; lane l owns the adjacent pairs P l .. P l +
// P - 1 (P = D / 64), so the halves x_i and x_{i + D/2} load as vectors.
//   inverse 0: dst[b][t] = R(pos) src[b][idx[t]]
//   inverse 1: dst[b][idx[t]] = R(pos)^T src[b][t]
// R(pos): (x_i, x_{i+D/2}) -> (x_i c - x_{i+D/2} s, x_{i+D/2} c + x_i s).
// ---------------------------------------------------------------------------
struct RopeArgs {
  double inv_freq[64];  // D/2 entries
};

template <typename T, int D>
__global__ void __launch_bounds__(256) permute_rope_kernel(const int32_t* __restrict__ idx,
                                                           const int32_t* __restrict__ cu, int32_t n_seqs,
                                                           int64_t seqlen, int64_t rows_total, int32_t heads,
                                                           const T* __restrict__ src, T* __restrict__ dst,
                                                           int inverse, const __grid_constant__ RopeArgs ra) {
  constexpr int P = D / 64;  // pairs per lane
  const int64_t warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows_total; row += warps) {
    const int64_t b = row / seqlen;
    const int64_t t = row - b * seqlen;
    const int32_t tok = idx[t];
    int32_t pos = tok;
    if (cu) {  // THD: position inside the sub-sequence holding tok
      int lo = 0, hi = n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
      }
      pos = tok - cu[lo];
    }
    float cs[P], sn[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const double ang = double(pos) * ra.inv_freq[lane * P + j];
      const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
      sincosf(float(red), &sn[j], &cs[j]);
      if (inverse) sn[j] = -sn[j];
    }
    const int64_t other = b * seqlen + tok;
    const int64_t s_row = inverse ? row : other;
    const int64_t d_row = inverse ? other : row;
    for (int h = 0; h < heads; ++h) {
      const T* ps = src + (s_row * heads + h) * D + lane * P;
      T* pd = dst + (d_row * heads + h) * D + lane * P;
      float x1[P], x2[P], y1[P], y2[P];
      load_vec<T, P>(ps, x1);
      load_vec<T, P>(ps + D / 2, x2);
#pragma unroll
      for (int j = 0; j < P; ++j) {
        y1[j] = x1[j] * cs[j] - x2[j] * sn[j];
        y2[j] = x2[j] * cs[j] + x1[j] * sn[j];
      }
      store_vec<T, P>(pd, y1);
      store_vec<T, P>(pd + D / 2, y2);
    }
  }
}

cp_status launch_permute_rope(const int32_t* idx, const int32_t* cu_dev, int32_t n_seqs, int32_t batch,
                              int64_t seqlen, int32_t heads, int32_t d, double base, const void* src, void* dst,
                              int inverse, cp_dtype dtype, cudaStream_t s) {
  if (d != 64 && d != 128) return CP_ERR_UNSUPPORTED;
  if (!(base > 0.0) || heads < 1) return CP_ERR_INVALID_ARG;
  RopeArgs ra{};
  for (int i = 0; i < d / 2; ++i) ra.inv_freq[i] = std::pow(base, -2.0 * i / d);
  const int64_t rows = int64_t(batch) * seqlen;
  if (rows == 0) return CP_OK;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > int64_t(num_sms()) * 16) blocks = int64_t(num_sms()) * 16;
  const int32_t* cu = cu_dev;
  if (dtype == CP_BF16) {
    auto* ps = static_cast<const __nv_bfloat16*>(src);
    auto* pd = static_cast<__nv_bfloat16*>(dst);
    if (d == 128)
      permute_rope_kernel<__nv_bfloat16, 128><<<unsigned(blocks), 256, 0, s>>>(idx, cu, n_seqs, seqlen, rows, heads,
                                                                             ps, pd, inverse, ra);
    else
      permute_rope_kernel<__nv_bfloat16, 64><<<unsigned(blocks), 256, 0, s>>>(idx, cu, n_seqs, seqlen, rows, heads,
                                                                            ps, pd, inverse, ra);
  } else {
    auto* ps = static_cast<const float*>(src);
    auto* pd = static_cast<float*>(dst);
    if (d == 128)
      permute_rope_kernel<float, 128><<<unsigned(blocks), 256, 0, s>>>(idx, cu, n_seqs, seqlen, rows, heads, ps, pd,
                                                                     inverse, ra);
    else
      permute_rope_kernel<float, 64><<<unsigned(blocks), 256, 0, s>>>(idx, cu, n_seqs, seqlen, rows, heads, ps, pd,
                                                                    inverse, ra);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
