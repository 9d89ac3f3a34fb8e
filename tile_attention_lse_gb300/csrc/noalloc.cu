// Ring forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: code that runs where
// cudaMalloc is forbidden or unavailable (inside an allocator callback, a
// plugin host that hands out only its own tensors, a pre-allocated serving
// process with a frozen memory budget).  cp_ring_attn_fwd_static_ws serves
// them with a workspace that lives in this library's own static device
// memory instead of a caller-provided buffer.
//
// The scratch is one file-scope array of kStaticWsBytes bytes in device
// memory; every GPU that loads the library holds it until the process exits.
// In host code the array's name is only a host-side stand-in, so its device
// address is obtained with cudaGetSymbolAddress on the first call made in
// each context (normally once per device, in its primary context).
#include <cuda.h>

#include <mutex>

#include "internal.h"
#include "plan.h"

namespace cpattn {
namespace {

constexpr size_t kStaticWsBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// The array's device address belongs to the context that loaded this
// library's device code, so the cache is keyed by the current context's
// unique id: a context created after cudaDeviceReset, or another context on
// the same device, looks the address up again instead of reusing a stale one.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CachedAddr {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
std::mutex g_static_mu;
CachedAddr g_static_cache[64];

template <typename F>
F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context; false when there is
// none (or the driver cannot tell).
bool current_ctx_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the static workspace in the current context: looked up
// on the first call in each context, with that context current, and cached
// under the context's id.  Where the driver cannot name the context the
// address is looked up on every call instead of being cached.
cp_status static_ws_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  unsigned long long id = 0;
  bool have_id = current_ctx_id(&id);
  CachedAddr& c = g_static_cache[dev];
  if (have_id && c.ptr && c.ctx_id == id) {
    *out = c.ptr;
    return CP_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return CP_ERR_CUDA;
  // the lookup makes the device's primary context current when none was
  if (!have_id) have_id = current_ctx_id(&id);
  c.ctx_id = have_id ? id : 0;
  c.ptr = have_id ? p : nullptr;
  *out = p;
  return CP_OK;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" size_t cp_static_ws_capacity(void) { return kStaticWsBytes; }

extern "C" cp_status cp_ring_attn_fwd_static_ws(const cp_attn_desc* desc, const void* q,
                                                const void* k, const void* v, void* o, float* lse,
                                                void* stream) {
  if (!desc) return CP_ERR_INVALID_ARG;
  cp_status st;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  if (!(desc->dtype == CP_F32 || (desc->dtype == CP_BF16 && desc->head_dim == 128)) ||
      (desc->dtype == CP_BF16 && !tc_available()))
    return CP_ERR_UNSUPPORTED;  // the same kernel rule as cp_ring_attn_fwd
  if (desc->seqlen == 0) return CP_OK;
  if (!q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(*desc, *p, false);
  if (w.total > kStaticWsBytes) return CP_ERR_WORKSPACE;  // problem too large for the static scratch
  void* ws = nullptr;
  st = static_ws_ptr(&ws);
  if (st != CP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  unsigned char* tables = base + w.tables;
  // Task-graph tables: copied from the plan's host image (pageable memory; no
  // pinned staging buffer is allocated on this path).  Every other byte of
  // the scratch is fully written by the kernels before it is read, so nothing
  // needs clearing between calls.
  if (!p->fwd_image.empty() &&
      cudaMemcpyAsync(tables, p->fwd_image.data(), p->fwd_image.size(), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return CP_ERR_CUDA;

  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_part = reinterpret_cast<float*>(base + w.part_o);
  a.lse_part = reinterpret_cast<float*>(base + w.part_l);
  a.o_out = o;
  a.lse_out = lse;
  a.items = reinterpret_cast<const TileItem*>(tables + p->off_fwd_items);
  a.segs = reinterpret_cast<const Seg*>(tables + p->off_fwd_segs);
  a.n_items = int32_t(p->fwd_items.size());
  a.wide_items = reinterpret_cast<const TileItem*>(tables + p->off_fwd_wide);
  a.wide_segs = reinterpret_cast<const Seg*>(tables + p->off_fwd_wide_segs);
  a.n_wide_items = int32_t(p->fwd_wide.size());
  a.batch = desc->batch;
  a.H = desc->heads_q;
  a.Hkv = desc->heads_kv;
  a.d = desc->head_dim;
  a.seqlen = desc->seqlen;
  a.part_rows = p->part_rows;
  a.scale = desc->softmax_scale > 0.0f ? desc->softmax_scale : 1.0f / sqrtf(float(desc->head_dim));
  a.causal = desc->causal;
  a.dtype = desc->dtype;
  if (a.n_items > 0) {
    ProfScope ps(CP_K_TILE_FWD, s);
    st = a.dtype == CP_BF16 ? launch_fwd_tc(a, s) : launch_fwd_simt(a, s);
    if (st != CP_OK) return st;
  }
  MergeArgs m{};
  m.o_part = a.o_part;
  m.lse_part = a.lse_part;
  m.o_out = o;
  m.lse_out = lse;
  m.segs = reinterpret_cast<const MergeSeg*>(tables + p->off_merge);
  m.n_segs = int32_t(p->merge_segs.size());
  m.merge_rows = p->merge_rows;
  m.batch = desc->batch;
  m.H = desc->heads_q;
  m.d = desc->head_dim;
  m.part_rows = p->part_rows;
  m.out_rows = desc->seqlen;
  m.out_dtype = desc->dtype;
  if (m.n_segs == 0) return CP_OK;  // every Q chunk was written by the forward itself
  ProfScope ps(CP_K_MERGE, s);
  return launch_merge(m, s);
}
