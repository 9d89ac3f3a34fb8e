// Partition index kernel and token gather ("04 · Megatron-LM 实现" §1.1:
// view as 2*cp chunks, rank r keeps chunks r and 2cp-1-r, then index_select;
// §1.2: the same inside every packed sub-sequence; "Context Parallelism (CP)"
// §4).
#include "internal.h"

namespace cpattn {

// One thread per rank-local slot g = r * (L / cp) + t.
//  BSHD (cu == nullptr): c = L / (2cp); slot t < c -> chunk r, else chunk 2cp-1-r.
//  THD: the rank's local stream is sub-sequence major; sub-sequence k occupies
//  local slots [cu[k] / cp, cu[k+1] / cp), front chunk then mirrored chunk.
__global__ void __launch_bounds__(256) partition_kernel(int32_t cp, int64_t L,
                                                        const int32_t* __restrict__ cu,
                                                        int32_t n_seqs, int32_t* __restrict__ idx,
                                                        int32_t* __restrict__ local_cu) {
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
  const int64_t chunk = off < c ? r : 2 * cp - 1 - r;
  const int64_t within = off < c ? off : off - c;
  idx[g] = int32_t(start + chunk * c + within);
}

cp_status launch_partition(int32_t cp, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                           int32_t* idx, int32_t* local_cu, cudaStream_t s) {
  const int64_t n = seqlen > n_seqs + 1 ? seqlen : n_seqs + 1;
  const unsigned blocks = unsigned((n + 255) / 256);
  partition_kernel<<<blocks, 256, 0, s>>>(cp, seqlen, cu_dev, n_seqs, idx, local_cu);
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
  if (blocks > 152 * 16) blocks = 152 * 16;
  permute_kernel<<<unsigned(blocks), 256, 0, s>>>(idx, seqlen, rows, row_bytes / 16,
                                                  static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst), inverse);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
