// CUDA-core (FFMA) tile attention, forward and backward, for float32 inputs
// (head_dim 64 or 128): a float32 input must meet 1e-5, which the tf32 and
// bf16 tensor-core paths cannot.  bf16 inputs run on the tcgen05 kernels
// only; these launchers refuse them.
//
// Forward ("Context Parallelism (CP)" §2.1, A_ij = TileAttention(...)): each
// thread block owns one work item (a Q tile of <= 128 rows and the K/V
// segments of one key owner) for one (batch, head); four threads share a
// query row, each holding a quarter of head_dim.  Keys stream through shared
// memory 32 at a time and the row state follows the online recurrence of
// "上下文并行" 02 ONE ROW: m' = max(m, max S), c = e^(m - m'), l' = c l + sum
// e^(S - m'), a' = c a + sum e^(S - m') V; the output is O = a / l and
// L = m + log l (natural log), or O = 0, L = -inf for a row that sees nothing.
//
// Backward ("上下文并行" 01 BACKWARD/REPLAY and GRADIENT/RETURN): P is
// rebuilt from the merged row LSE, dS = P (dP - D).  dQ is computed per Q tile
// over every visible K/V range; dK and dV per K/V tile over every Q range of
// every query rank (and every q-head of the group), which is the sum at the
// key owner.  No atomics: each output row is written by exactly one block.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "internal.h"

namespace cpattn {

namespace {

struct ItemView {
  int32_t row0, pos0, len, out_row0, seg_count;
  const Seg* segs;
  Seg single;
};

__device__ __forceinline__ ItemView fwd_item(const FwdArgs& a, int i) {
  ItemView v;
  if (a.items) {
    const TileItem it = a.items[i];
    v.row0 = it.row0;
    v.pos0 = it.pos0;
    v.len = it.len;
    v.out_row0 = it.out_row0;
    v.seg_count = it.seg_count;
    v.segs = a.segs + it.seg_begin;
  } else {
    v.row0 = a.edge.q_row0 + i * kTile;
    v.pos0 = a.edge.q_pos0 + i * kTile;
    v.len = min(kTile, a.edge.q_len - i * kTile);
    v.out_row0 = i * kTile;
    v.seg_count = 1;
    v.single = Seg{a.edge.kv_row0, a.edge.kv_pos0, a.edge.kv_len, a.edge.win};
    v.segs = nullptr;
  }
  return v;
}

template <int TPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = 1; o < TPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kFwdThreads = 512;  // 128 rows x 4 threads
constexpr int kFwdTPR = 4;
constexpr int kFwdBK = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kFwdThreads) fwd_simt_kernel(FwdArgs a) {
  constexpr int TPR = kFwdTPR;
  constexpr int NG = D / 4 / TPR;  // float4 groups per thread
  constexpr int BK = kFwdBK;
  __shared__ __align__(16) float sK[BK][D];
  __shared__ __align__(16) float sV[BK][D];

  const int tid = threadIdx.x;
  const int row = tid / TPR, part = tid % TPR;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (a.H / a.Hkv);
  const ItemView it = fwd_item(a, blockIdx.x);
  const bool active = row < it.len;
  const int qpos = it.pos0 + row;
  const int64_t S = a.seqlen;

  float q[NG * 4], o[NG * 4];
  {
    const T* qp = static_cast<const T*>(a.q) + ((int64_t(b) * S + it.row0 + (active ? row : 0)) * a.H + h) * D;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      load_vec<T, 4>(qp + 4 * (part + TPR * j), &q[4 * j]);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        q[4 * j + t] = active ? q[4 * j + t] * a.scale : 0.f;
        o[4 * j + t] = 0.f;
      }
    }
  }
  float m = -INFINITY, l = 0.f;
  const int qlast = it.pos0 + it.len - 1;

  for (int si = 0; si < it.seg_count; ++si) {
    const Seg sg = it.segs ? it.segs[si] : it.single;
    int eff = sg.len;
    if (a.causal) eff = min(eff, qlast - sg.pos0 + 1);
    for (int kt = 0; kt < eff; kt += BK) {
      __syncthreads();
      for (int e = tid; e < BK * D / 4; e += kFwdThreads) {
        const int j = e / (D / 4), c4 = e % (D / 4);
        float kk[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
        if (kt + j < eff) {
          const int64_t off = ((int64_t(b) * S + sg.row0 + kt + j) * a.Hkv + g) * D + 4 * c4;
          load_vec<T, 4>(static_cast<const T*>(a.k) + off, kk);
          load_vec<T, 4>(static_cast<const T*>(a.v) + off, vv);
        }
        *reinterpret_cast<float4*>(&sK[j][4 * c4]) = make_float4(kk[0], kk[1], kk[2], kk[3]);
        *reinterpret_cast<float4*>(&sV[j][4 * c4]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
      }
      __syncthreads();
      float sc[BK];
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < BK; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const float4 kv = *reinterpret_cast<const float4*>(&sK[j][4 * (part + TPR * gi)]);
          acc = fmaf(q[4 * gi], kv.x, acc);
          acc = fmaf(q[4 * gi + 1], kv.y, acc);
          acc = fmaf(q[4 * gi + 2], kv.z, acc);
          acc = fmaf(q[4 * gi + 3], kv.w, acc);
        }
        acc = group_sum<TPR>(acc);
        const bool vis = active && (kt + j < eff) && (!a.causal || sg.pos0 + kt + j <= qpos) &&
                         (sg.win == 0 || qpos - (sg.pos0 + kt + j) < sg.win);
        sc[j] = vis ? acc : -INFINITY;
        tmax = fmaxf(tmax, sc[j]);
      }
      const float m_new = fmaxf(m, tmax);
      if (m_new == -INFINITY) continue;  // nothing visible yet for this row
      const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
      l *= corr;
#pragma unroll
      for (int t = 0; t < NG * 4; ++t) o[t] *= corr;
#pragma unroll
      for (int j = 0; j < BK; ++j) {
        const float p = expf(sc[j] - m_new);  // 0 for masked keys
        l += p;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const float4 vv = *reinterpret_cast<const float4*>(&sV[j][4 * (part + TPR * gi)]);
          o[4 * gi] = fmaf(p, vv.x, o[4 * gi]);
          o[4 * gi + 1] = fmaf(p, vv.y, o[4 * gi + 1]);
          o[4 * gi + 2] = fmaf(p, vv.z, o[4 * gi + 2]);
          o[4 * gi + 3] = fmaf(p, vv.w, o[4 * gi + 3]);
        }
      }
      m = m_new;
    }
  }
  if (!active) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  // a single-part Q chunk (out_row0 = -1) is final here: O in the input
  // type and LSE go to the outputs at the item's own rows
  const bool direct = it.out_row0 < 0;
  const int64_t prow = direct ? int64_t(b) * S + it.row0 + row : int64_t(b) * a.part_rows + it.out_row0 + row;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    float x[4] = {o[4 * gi] * inv, o[4 * gi + 1] * inv, o[4 * gi + 2] * inv, o[4 * gi + 3] * inv};
    if (direct)
      store_vec<T, 4>(static_cast<T*>(a.o_out) + (prow * a.H + h) * D + 4 * (part + TPR * gi), x);
    else
      store_vec<float, 4>(a.o_part + (prow * a.H + h) * D + 4 * (part + TPR * gi), x);
  }
  if (part == 0) (direct ? a.lse_out : a.lse_part)[prow * a.H + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ----------------------------- backward: dQ --------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kFwdThreads) bwd_dq_simt_kernel(BwdArgs a) {
  constexpr int TPR = kFwdTPR;
  constexpr int NG = D / 4 / TPR;
  constexpr int BK = kFwdBK;
  __shared__ __align__(16) float sK[BK][D];
  __shared__ __align__(16) float sV[BK][D];
  const int tid = threadIdx.x;
  const int row = tid / TPR, part = tid % TPR;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (a.H / a.Hkv);
  const TileItem it = a.q_items[blockIdx.x];
  const bool active = row < it.len;
  const int qpos = it.pos0 + row;
  const int64_t S = a.seqlen;
  const int64_t qrow = int64_t(b) * S + it.row0 + (active ? row : 0);

  float q[NG * 4], dob[NG * 4], dq[NG * 4];
  {
    const T* qp = static_cast<const T*>(a.q) + (qrow * a.H + h) * D;
    const T* dp = static_cast<const T*>(a.dout) + (qrow * a.H + h) * D;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      load_vec<T, 4>(qp + 4 * (part + TPR * j), &q[4 * j]);
      load_vec<T, 4>(dp + 4 * (part + TPR * j), &dob[4 * j]);
#pragma unroll
      for (int t = 0; t < 4; ++t) dq[4 * j + t] = 0.f;
    }
  }
  const float L = a.lse[qrow * a.H + h];
  const float Dl = a.delta[(int64_t(b) * a.H + h) * S + it.row0 + (active ? row : 0)];
  const bool live = active && L != -INFINITY;
  const int qlast = it.pos0 + it.len - 1;
  for (int si = 0; si < it.seg_count; ++si) {
    const Seg sg = a.q_segs[it.seg_begin + si];
    int eff = sg.len;
    if (a.causal) eff = min(eff, qlast - sg.pos0 + 1);
    for (int kt = 0; kt < eff; kt += BK) {
      __syncthreads();
      for (int e = tid; e < BK * D / 4; e += kFwdThreads) {
        const int j = e / (D / 4), c4 = e % (D / 4);
        float kk[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
        if (kt + j < eff) {
          const int64_t off = ((int64_t(b) * S + sg.row0 + kt + j) * a.Hkv + g) * D + 4 * c4;
          load_vec<T, 4>(static_cast<const T*>(a.k) + off, kk);
          load_vec<T, 4>(static_cast<const T*>(a.v) + off, vv);
        }
        *reinterpret_cast<float4*>(&sK[j][4 * c4]) = make_float4(kk[0], kk[1], kk[2], kk[3]);
        *reinterpret_cast<float4*>(&sV[j][4 * c4]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
      }
      __syncthreads();
#pragma unroll 4
      for (int j = 0; j < BK; ++j) {
        float s = 0.f, dpv = 0.f;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const float4 kv = *reinterpret_cast<const float4*>(&sK[j][4 * (part + TPR * gi)]);
          const float4 vv = *reinterpret_cast<const float4*>(&sV[j][4 * (part + TPR * gi)]);
          s = fmaf(q[4 * gi], kv.x, s); s = fmaf(q[4 * gi + 1], kv.y, s);
          s = fmaf(q[4 * gi + 2], kv.z, s); s = fmaf(q[4 * gi + 3], kv.w, s);
          dpv = fmaf(dob[4 * gi], vv.x, dpv); dpv = fmaf(dob[4 * gi + 1], vv.y, dpv);
          dpv = fmaf(dob[4 * gi + 2], vv.z, dpv); dpv = fmaf(dob[4 * gi + 3], vv.w, dpv);
        }
        s = group_sum<TPR>(s);
        dpv = group_sum<TPR>(dpv);
        const bool vis = live && (kt + j < eff) && (!a.causal || sg.pos0 + kt + j <= qpos) &&
                         (sg.win == 0 || qpos - (sg.pos0 + kt + j) < sg.win);
        const float p = vis ? expf(s * a.scale - L) : 0.f;
        const float ds = p * (dpv - Dl);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          const float4 kv = *reinterpret_cast<const float4*>(&sK[j][4 * (part + TPR * gi)]);
          dq[4 * gi] = fmaf(ds, kv.x, dq[4 * gi]);
          dq[4 * gi + 1] = fmaf(ds, kv.y, dq[4 * gi + 1]);
          dq[4 * gi + 2] = fmaf(ds, kv.z, dq[4 * gi + 2]);
          dq[4 * gi + 3] = fmaf(ds, kv.w, dq[4 * gi + 3]);
        }
      }
    }
  }
  if (!active) return;
  T* out = static_cast<T*>(a.dq) + (qrow * a.H + h) * D;
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    float x[4] = {dq[4 * gi] * a.scale, dq[4 * gi + 1] * a.scale, dq[4 * gi + 2] * a.scale,
                  dq[4 * gi + 3] * a.scale};
    store_vec<T, 4>(out + 4 * (part + TPR * gi), x);
  }
}

// --------------------------- backward: dK, dV -------------------------------
constexpr int kKvThreads = 512;  // 64 key rows x 8 threads per pass
constexpr int kKvTPR = 8;
constexpr int kKvRows = 64;
constexpr int kKvBQ = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kKvThreads) bwd_dkdv_simt_kernel(BwdArgs a) {
  constexpr int TPR = kKvTPR;
  constexpr int NG = D / 4 / TPR;
  constexpr int BQ = kKvBQ;
  __shared__ __align__(16) float sQ[BQ][D];
  __shared__ __align__(16) float sO[BQ][D];  // dO rows
  __shared__ float sL[BQ], sD[BQ];
  const int tid = threadIdx.x;
  const int rrow = tid / TPR, part = tid % TPR;
  const int g = blockIdx.y, b = blockIdx.z;
  const int group = a.H / a.Hkv;
  const TileItem it = a.kv_items[blockIdx.x];
  const int64_t S = a.seqlen;

  for (int pass = 0; pass * kKvRows < it.len; ++pass) {
    const int r = pass * kKvRows + rrow;
    const bool active = r < it.len;
    const int kpos = it.pos0 + r;
    const int64_t krow = int64_t(b) * S + it.row0 + (active ? r : 0);
    float kk[NG * 4], vv[NG * 4], dk[NG * 4], dv[NG * 4];
    {
      const T* kp = static_cast<const T*>(a.k) + (krow * a.Hkv + g) * D;
      const T* vp = static_cast<const T*>(a.v) + (krow * a.Hkv + g) * D;
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        load_vec<T, 4>(kp + 4 * (part + TPR * j), &kk[4 * j]);
        load_vec<T, 4>(vp + 4 * (part + TPR * j), &vv[4 * j]);
#pragma unroll
        for (int t = 0; t < 4; ++t) { dk[4 * j + t] = 0.f; dv[4 * j + t] = 0.f; }
      }
    }
    for (int hj = 0; hj < group; ++hj) {
      const int h = g * group + hj;
      for (int si = 0; si < it.seg_count; ++si) {
        const Seg sg = a.kv_segs[it.seg_begin + si];
        for (int qt = 0; qt < sg.len; qt += BQ) {
          __syncthreads();
          for (int e = tid; e < BQ * D / 4; e += kKvThreads) {
            const int i = e / (D / 4), c4 = e % (D / 4);
            float xq[4] = {0.f, 0.f, 0.f, 0.f}, xo[4] = {0.f, 0.f, 0.f, 0.f};
            if (qt + i < sg.len) {
              const int64_t off = ((int64_t(b) * S + sg.row0 + qt + i) * a.H + h) * D + 4 * c4;
              load_vec<T, 4>(static_cast<const T*>(a.q) + off, xq);
              load_vec<T, 4>(static_cast<const T*>(a.dout) + off, xo);
            }
            *reinterpret_cast<float4*>(&sQ[i][4 * c4]) = make_float4(xq[0], xq[1], xq[2], xq[3]);
            *reinterpret_cast<float4*>(&sO[i][4 * c4]) = make_float4(xo[0], xo[1], xo[2], xo[3]);
          }
          if (tid < BQ) {
            float lv = -INFINITY, dl = 0.f;
            if (qt + tid < sg.len) {
              const int64_t rr = (int64_t(b) * S + sg.row0 + qt + tid) * a.H + h;
              lv = a.lse[rr];
              dl = a.delta[(int64_t(b) * a.H + h) * S + sg.row0 + qt + tid];
            }
            sL[tid] = lv;
            sD[tid] = dl;
          }
          __syncthreads();
#pragma unroll 4
          for (int i = 0; i < BQ; ++i) {
            float s = 0.f, dpv = 0.f;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
              const float4 xq = *reinterpret_cast<const float4*>(&sQ[i][4 * (part + TPR * gi)]);
              const float4 xo = *reinterpret_cast<const float4*>(&sO[i][4 * (part + TPR * gi)]);
              s = fmaf(kk[4 * gi], xq.x, s); s = fmaf(kk[4 * gi + 1], xq.y, s);
              s = fmaf(kk[4 * gi + 2], xq.z, s); s = fmaf(kk[4 * gi + 3], xq.w, s);
              dpv = fmaf(vv[4 * gi], xo.x, dpv); dpv = fmaf(vv[4 * gi + 1], xo.y, dpv);
              dpv = fmaf(vv[4 * gi + 2], xo.z, dpv); dpv = fmaf(vv[4 * gi + 3], xo.w, dpv);
            }
            s = group_sum<TPR>(s);
            dpv = group_sum<TPR>(dpv);
            const float Li = sL[i];
            const bool vis = active && (qt + i < sg.len) && Li != -INFINITY &&
                             (!a.causal || kpos <= sg.pos0 + qt + i) &&
                             (sg.win == 0 || sg.pos0 + qt + i - kpos < sg.win);
            const float p = vis ? expf(s * a.scale - Li) : 0.f;
            const float ds = p * (dpv - sD[i]);
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
              const float4 xq = *reinterpret_cast<const float4*>(&sQ[i][4 * (part + TPR * gi)]);
              const float4 xo = *reinterpret_cast<const float4*>(&sO[i][4 * (part + TPR * gi)]);
              dv[4 * gi] = fmaf(p, xo.x, dv[4 * gi]); dv[4 * gi + 1] = fmaf(p, xo.y, dv[4 * gi + 1]);
              dv[4 * gi + 2] = fmaf(p, xo.z, dv[4 * gi + 2]); dv[4 * gi + 3] = fmaf(p, xo.w, dv[4 * gi + 3]);
              dk[4 * gi] = fmaf(ds, xq.x, dk[4 * gi]); dk[4 * gi + 1] = fmaf(ds, xq.y, dk[4 * gi + 1]);
              dk[4 * gi + 2] = fmaf(ds, xq.z, dk[4 * gi + 2]); dk[4 * gi + 3] = fmaf(ds, xq.w, dk[4 * gi + 3]);
            }
          }
        }
      }
    }
    if (active) {
      T* pk = static_cast<T*>(a.dk) + (krow * a.Hkv + g) * D;
      T* pv = static_cast<T*>(a.dv) + (krow * a.Hkv + g) * D;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float xk[4] = {dk[4 * gi] * a.scale, dk[4 * gi + 1] * a.scale, dk[4 * gi + 2] * a.scale,
                       dk[4 * gi + 3] * a.scale};
        store_vec<T, 4>(pk + 4 * (part + TPR * gi), xk);
        store_vec<T, 4>(pv + 4 * (part + TPR * gi), &dv[4 * gi]);
      }
    }
  }
}

}  // namespace

cp_status launch_fwd_simt(const FwdArgs& a, cudaStream_t s) {
  if (a.dtype != CP_F32) return CP_ERR_UNSUPPORTED;  // bf16 runs on the tcgen05 kernels only
  if (a.n_items == 0) return CP_OK;
  const dim3 grid(unsigned(a.n_items), unsigned(a.H), unsigned(a.batch));
  if (a.d == 128) fwd_simt_kernel<float, 128><<<grid, kFwdThreads, 0, s>>>(a);
  else fwd_simt_kernel<float, 64><<<grid, kFwdThreads, 0, s>>>(a);
  return cuda_status(cudaGetLastError());
}

cp_status launch_bwd_simt(const BwdArgs& a, cudaStream_t s) {
  if (a.dtype != CP_F32) return CP_ERR_UNSUPPORTED;
  if (a.n_q_items > 0) {
    const dim3 grid(unsigned(a.n_q_items), unsigned(a.H), unsigned(a.batch));
    if (a.d == 128) bwd_dq_simt_kernel<float, 128><<<grid, kFwdThreads, 0, s>>>(a);
    else bwd_dq_simt_kernel<float, 64><<<grid, kFwdThreads, 0, s>>>(a);
    const cp_status st = cuda_status(cudaGetLastError());
    if (st != CP_OK) return st;
  }
  if (a.n_kv_items > 0) {
    const dim3 grid(unsigned(a.n_kv_items), unsigned(a.Hkv), unsigned(a.batch));
    if (a.d == 128) bwd_dkdv_simt_kernel<float, 128><<<grid, kKvThreads, 0, s>>>(a);
    else bwd_dkdv_simt_kernel<float, 64><<<grid, kKvThreads, 0, s>>>(a);
    return cuda_status(cudaGetLastError());
  }
  return CP_OK;
}

}  // namespace cpattn
