// Small memory-bound kernels shared by the forward and backward paths, and the
// device error word.
#include <cuda_bf16.h>

#include <atomic>

#include "device_util.cuh"
#include "internal.h"
#include "tmap.h"
#include "tc_util.cuh"

namespace cpattn {

__device__ int g_cp_device_error = 0;

namespace {
std::atomic<long long> g_wait_limit{tc::kWaitCycles};
}  // namespace

long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

// Kernels of other translation units receive the word's address as an
// argument (no relocatable device code needed).
int* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  // per device; host threads may race on the first lookup, which every one
  // of them makes the same way
  static std::atomic<int*> cached[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  int* c = cached[dev].load(std::memory_order_acquire);
  if (!c) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cp_device_error) != cudaSuccess) return nullptr;
    c = static_cast<int*>(p);
    cached[dev].store(c, std::memory_order_release);
  }
  return c;
}

cp_status set_wait_limit_cycles(int64_t cycles) {
  if (cycles > tc::kWaitCycles) return CP_ERR_INVALID_ARG;
  g_wait_limit.store(cycles <= 0 ? tc::kWaitCycles : static_cast<long long>(cycles), std::memory_order_relaxed);
  return CP_OK;
}

cp_status read_and_clear_device_error(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return CP_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_cp_device_error, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_cp_device_error, &zero, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    return CP_ERR_TIMEOUT;
  }
  return CP_OK;
}

// ---------------------------------------------------------------------------
// Backward preprocess ("上下文并行" 01 BACKWARD/REPLAY: the replay uses the
// full-row LSE and the output): per (row, head)
//   D  = <dO, O>                         float32, head-major [b][h][s]
//   L2 = lse * log2(e)  (+inf if the row saw no key, so exp2(S - L2) = 0)
// 16-byte vectors: a warp covers 1 to 4 (row, head)s per load, lanes split head_dim.
// The same grid also zeroes the tensor-core path's dQ accumulator: when it
// holds 128 floats per (row, head), the warp that reads a group of (row,
// head)s writes the zeros of as many accumulator rows in the same step, so
// the reads and the writes share the memory system instead of following one
// another; any other size is zeroed by a grid-stride loop first.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const T* __restrict__ o,
                                                       const T* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ delta,
                                                       float* __restrict__ lse2, int64_t S, int H,
                                                       int64_t n_rowheads, float4* __restrict__ zero,
                                                       int64_t n_zero4) {
  // 16-byte vectors: a row of head_dim elements spans kLanes lanes, so one
  // warp-wide load covers kRows rows; two such groups are in flight per step.
  constexpr int kVec = 16 / int(sizeof(T));
  constexpr int kLanes = D / kVec;
  constexpr int kRows = 32 / kLanes;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanes, sl = lane - sub * kLanes;
  const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t n_threads = int64_t(gridDim.x) * blockDim.x;
  const bool zero_with_rows = n_zero4 == n_rowheads * 32;  // 128 floats per (row, head)
  if (!zero_with_rows)
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_zero4; i += n_threads)
      zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t r0 = warp * 2 * kRows; r0 < n_rowheads; r0 += n_warps * 2 * kRows) {
    if (zero_with_rows) {  // accumulator rows r0 .. r0 + 2 kRows - 1: 512 bytes each
#pragma unroll
      for (int u = 0; u < 2 * kRows; ++u)
        if (r0 + u < n_rowheads) zero[(r0 + u) * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc[2] = {0.f, 0.f};
    float a[2][kVec], b[2][kVec];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t rh = r0 + u * kRows + sub;
      if (rh < n_rowheads) {
        load_vec<T, kVec>(o + rh * D + sl * kVec, a[u]);
        load_vec<T, kVec>(dout + rh * D + sl * kVec, b[u]);
      } else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) a[u][i] = b[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[u] = fmaf(a[u][i], b[u][i], acc[u]);
#pragma unroll
      for (int off = kLanes / 2; off > 0; off >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
      const int64_t rh = r0 + u * kRows + sub;
      if (sl == 0 && rh < n_rowheads) {
        const int h = int(rh % H);
        const int64_t br = rh / H;
        const int64_t bb = br / S, row = br - bb * S;
        const int64_t t = (bb * H + h) * S + row;
        delta[t] = acc[u];
        const float l = lse[rh];
        lse2[t] = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;
      }
    }
  }
}

cp_status launch_bwd_prep(const void* o, const void* dout, const float* lse, float* delta,
                          float* lse2, int32_t batch, int64_t S, int32_t H, int32_t d,
                          cp_dtype dtype, float* zero, int64_t zero_floats, cudaStream_t s) {
  const int64_t n = int64_t(batch) * S * H;
  if (n == 0) return CP_OK;
  if (zero_floats % 4 != 0 || (reinterpret_cast<uintptr_t>(zero) & 15) != 0) return CP_ERR_ALIGNMENT;
  float4* z4 = reinterpret_cast<float4*>(zero);
  const int64_t nz4 = zero ? zero_floats / 4 : 0;
  const int threads = 256;
  int64_t blocks = (n + 31) / 32;  // up to 32 row-heads per 8-warp block per step
  const int64_t cap8 = int64_t(num_sms()) * 8;
  blocks = blocks > cap8 ? cap8 : blocks;
  const dim3 g(static_cast<unsigned>(blocks));
  if (dtype == CP_BF16) {
    auto* po = static_cast<const __nv_bfloat16*>(o);
    auto* pd = static_cast<const __nv_bfloat16*>(dout);
    if (d == 128) bwd_prep_kernel<__nv_bfloat16, 128><<<g, threads, 0, s>>>(po, pd, lse, delta, lse2, S, H, n, z4, nz4);
    else bwd_prep_kernel<__nv_bfloat16, 64><<<g, threads, 0, s>>>(po, pd, lse, delta, lse2, S, H, n, z4, nz4);
  } else {
    auto* po = static_cast<const float*>(o);
    auto* pd = static_cast<const float*>(dout);
    if (d == 128) bwd_prep_kernel<float, 128><<<g, threads, 0, s>>>(po, pd, lse, delta, lse2, S, H, n, z4, nz4);
    else bwd_prep_kernel<float, 64><<<g, threads, 0, s>>>(po, pd, lse, delta, lse2, S, H, n, z4, nz4);
  }
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Task-graph tables: device-mapped pinned host memory -> workspace, 16 bytes
// per thread and step (the reads cross the host link; the tables are small).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                     int64_t n16) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

cp_status launch_copy_from_host(void* dst, const void* src_mapped, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return CP_OK;
  if ((bytes & 15) != 0 || ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src_mapped)) & 15) != 0)
    return CP_ERR_ALIGNMENT;
  const int64_t n16 = int64_t(bytes / 16);
  int64_t blocks = (n16 + 255) / 256;
  const int64_t cap4 = int64_t(num_sms()) * 4;
  blocks = blocks > cap4 ? cap4 : blocks;
  copy16_kernel<<<unsigned(blocks), 256, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src_mapped),
                                                  n16);
  return cuda_status(cudaGetLastError());
}

}  // namespace cpattn
