// extern "C" boundary of libcpattn: argument validation, workspace layout,
// table upload and kernel launches on the caller's stream.  No entry point
// allocates device memory.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "plan.h"

using namespace cpattn;

namespace {

size_t elem_bytes(cp_dtype t) { return t == CP_BF16 ? 2 : 4; }

float eff_scale(const cp_attn_desc& d) {
  return d.softmax_scale > 0.0f ? d.softmax_scale : 1.0f / std::sqrt(float(d.head_dim));
}

// Copies a plan's table image into the workspace from pinned, device-mapped
// host memory with a small kernel on the caller's stream (the pinned image is
// immutable once built).  A kernel rather than a copy-engine transfer, so the
// upload never queues behind the caller's own host<->device copies.
cp_status upload(void* dst, const std::vector<unsigned char>& img, void** pinned,
                 cudaStream_t s);

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255) == 0; }

// The attention kernels are fixed by the element type, never chosen at run
// time: float32 runs on the FFMA kernels (float32 arithmetic throughout, the
// only way to the float32 bar), bf16 on the tcgen05 kernels, which are built
// for head_dim 128.  bf16 at any other head_dim, or a driver without the
// tensor-map encoder the tcgen05 kernels need, is refused.
bool attn_shape_built(const cp_attn_desc& d) {
  return d.dtype == CP_F32 || (d.dtype == CP_BF16 && d.head_dim == 128);
}
cp_status attn_kernels_for(const cp_attn_desc& d) {
  if (!attn_shape_built(d)) return CP_ERR_UNSUPPORTED;
  if (d.dtype == CP_BF16 && !tc_available()) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

// ---- benchmark instrumentation: events around every launch when enabled ----
struct ProfRecord {
  int kid;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;
int64_t g_prof_launches[CP_K_COUNT] = {};

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

cp_status upload(void* dst, const std::vector<unsigned char>& img, void** pinned,
                 cudaStream_t s) {
  if (img.empty()) return CP_OK;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!*pinned) {
      void* h = nullptr;
      if (cudaHostAlloc(&h, img.size(), cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
        return CP_ERR_CUDA;
      std::memcpy(h, img.data(), img.size());
      *pinned = h;
    }
  }
  void* src = nullptr;
  if (cudaHostGetDevicePointer(&src, *pinned, 0) != cudaSuccess) return CP_ERR_CUDA;
  ProfScope ps(CP_K_TABLES, s);
  return launch_copy_from_host(dst, src, img.size(), s);
}

}  // namespace

namespace cpattn {

ProfScope::ProfScope(int kernel_class, cudaStream_t s, int n_launches) : kid_(kernel_class), s_(s) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_launches[kid_] += n_launches;
  if (g_prof_on) {
    a_ = prof_event();
    b_ = prof_event();
    if (a_ && b_) cudaEventRecord(a_, s_);
  }
}

ProfScope::~ProfScope() {
  if (!a_ || !b_) return;
  cudaEventRecord(b_, s_);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_recs.push_back(ProfRecord{kid_, a_, b_});
}

}  // namespace cpattn

extern "C" {

const char* cp_status_string(cp_status st) {
  switch (st) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_ALIGNMENT: return "CP_ERR_ALIGNMENT";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT";
  }
  return "CP_ERR_UNKNOWN";
}

cp_status cp_validate_desc(const cp_attn_desc* desc) { return validate(desc); }

cp_status cp_ring_plan_stats(const cp_attn_desc* desc, int64_t out[6]) {
  if (!out) return CP_ERR_INVALID_ARG;
  cp_status st;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  out[0] = int64_t(p->fwd_items.size());
  out[1] = p->part_rows;
  out[2] = int64_t(p->merge_segs.size());
  out[3] = int64_t(p->kv_items.size());
  out[4] = p->pairs;
  out[5] = p->fwd_tiles;
  return CP_OK;
}

cp_status cp_ring_plan_tables(const cp_attn_desc* desc, int32_t which, int64_t* n_items, int64_t* n_segs,
                              int32_t* items, int32_t* segs) {
  if (!desc || which < 0 || which > 4) return CP_ERR_INVALID_ARG;
  cp_status st;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  if (which == 4) {  // merge segments
    if (n_items) *n_items = int64_t(p->merge_segs.size());
    if (n_segs) *n_segs = 0;
    for (size_t i = 0; items && i < p->merge_segs.size(); ++i) {
      const MergeSeg& m = p->merge_segs[i];
      const int32_t row[8] = {m.out_row0, m.len, m.part_row0, m.n_parts, m.part_stride, m.merge_row0, 0, 0};
      std::copy(row, row + 8, items + 8 * i);
    }
    return CP_OK;
  }
  const std::vector<TileItem>* it[4] = {&p->fwd_items, &p->fwd_wide, &p->kv_items, &p->q_items};
  const std::vector<Seg>* sg[4] = {&p->fwd_segs, &p->fwd_wide_segs, &p->kv_segs, &p->q_segs};
  const auto& I = *it[which];
  const auto& S = *sg[which];
  if (n_items) *n_items = int64_t(I.size());
  if (n_segs) *n_segs = int64_t(S.size());
  for (size_t i = 0; items && i < I.size(); ++i) {
    const TileItem& t = I[i];
    const int32_t row[8] = {t.row0, t.pos0, t.len, t.seg_begin, t.seg_count, t.out_row0, t.cost, 0};
    std::copy(row, row + 8, items + 8 * i);
  }
  for (size_t i = 0; segs && i < S.size(); ++i) {
    const int32_t row[4] = {S[i].row0, S[i].pos0, S[i].len, S[i].win};
    std::copy(row, row + 4, segs + 4 * i);
  }
  return CP_OK;
}

cp_status cp_ring_bwd_schedule(const cp_attn_desc* desc, int32_t* grid, int64_t* n_work, int32_t* cta,
                               int32_t* work, int64_t* load) {
  if (!desc) return CP_ERR_INVALID_ARG;
  cp_status st;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  if (grid) *grid = p->kv_grid;
  if (n_work) *n_work = int64_t(p->kv_work.size());
  if (cta) std::copy(p->kv_cta.begin(), p->kv_cta.end(), cta);
  if (work) std::copy(p->kv_work.begin(), p->kv_work.end(), work);
  if (load) {
    const int64_t n_items = int64_t(p->kv_items.size());
    const int group = desc->heads_q / desc->heads_kv;
    for (int32_t c = 0; c < p->kv_grid; ++c) {
      int64_t sum = 0;
      for (int32_t k = p->kv_cta[size_t(c)]; k < p->kv_cta[size_t(c) + 1]; ++k)
        sum += int64_t(p->kv_items[size_t(p->kv_work[size_t(k)] % n_items)].cost) * group + 1;
      load[c] = sum;
    }
  }
  return CP_OK;
}

size_t cp_ring_attn_workspace_bytes(const cp_attn_desc* desc, int32_t backward) {
  if (!desc) return 0;
  cp_status st;
  auto p = get_plan(*desc, &st);
  if (!p || !attn_shape_built(*desc)) return 0;
  return ws_layout(*desc, *p, backward != 0).total;
}

cp_status cp_partition_indices(const cp_attn_desc* desc, int32_t* idx, int32_t* local_cu,
                               void* stream) {
  cp_status st = validate(desc);
  if (st != CP_OK) return st;
  if (desc->seqlen == 0) return CP_OK;
  if (!idx) return CP_ERR_INVALID_ARG;
  const bool thd = desc->cu_seqlens_host != nullptr;
  if (thd && !desc->cu_seqlens_dev) return CP_ERR_INVALID_ARG;
  if (!thd && local_cu) return CP_ERR_INVALID_ARG;
  ProfScope ps(CP_K_PARTITION, static_cast<cudaStream_t>(stream));
  if (desc->seq_cp_host) {  // hybrid CP: per-rank slice table required
    if (!local_cu || !desc->seq_cp_dev || !desc->seq_rank0_dev) return CP_ERR_INVALID_ARG;
    return launch_partition_hybrid(desc->cp, desc->seqlen, desc->cu_seqlens_dev, desc->n_seqs, desc->seq_cp_dev,
                                   desc->seq_rank0_dev, idx, local_cu, static_cast<cudaStream_t>(stream));
  }
  return launch_partition(desc->cp, desc->seqlen, thd ? desc->cu_seqlens_dev : nullptr,
                          thd ? desc->n_seqs : 0, idx, local_cu, desc->partition == CP_PARTITION_STRIPED,
                          static_cast<cudaStream_t>(stream));
}

cp_status cp_token_seq_pos(const cp_attn_desc* desc, const int32_t* idx, int32_t* seq_pos, void* stream) {
  cp_status st = validate(desc);
  if (st != CP_OK) return st;
  if (desc->seqlen == 0) return CP_OK;
  if (!idx || !seq_pos) return CP_ERR_INVALID_ARG;
  const bool thd = desc->cu_seqlens_host != nullptr;
  if (thd && (!desc->cu_seqlens_dev || desc->n_seqs < 1)) return CP_ERR_INVALID_ARG;
  ProfScope ps(CP_K_PARTITION, static_cast<cudaStream_t>(stream));
  return launch_token_seq_pos(idx, desc->seqlen, thd ? desc->cu_seqlens_dev : nullptr, thd ? desc->n_seqs : 0,
                              seq_pos, static_cast<cudaStream_t>(stream));
}

cp_status cp_permute_tokens(const cp_attn_desc* desc, const int32_t* idx, int32_t heads,
                            const void* src, void* dst, int32_t inverse, void* stream) {
  cp_status st = validate(desc);
  if (st != CP_OK) return st;
  if (heads < 1) return CP_ERR_INVALID_ARG;
  if (desc->seqlen == 0) return CP_OK;
  if (!idx || !src || !dst || src == dst) return CP_ERR_INVALID_ARG;
  const int64_t row_bytes = int64_t(heads) * desc->head_dim * elem_bytes(desc->dtype);
  ProfScope ps(CP_K_PERMUTE, static_cast<cudaStream_t>(stream));
  return launch_permute(idx, desc->batch, desc->seqlen, row_bytes, src, dst, inverse != 0,
                        static_cast<cudaStream_t>(stream));
}

cp_status cp_permute_rope(const cp_attn_desc* desc, const int32_t* idx, int32_t heads, float rope_base,
                          const void* src, void* dst, int32_t inverse, void* stream) {
  cp_status st = validate(desc);
  if (st != CP_OK) return st;
  if (heads < 1 || !(rope_base > 0.f)) return CP_ERR_INVALID_ARG;
  if (desc->seqlen == 0) return CP_OK;
  if (!idx || !src || !dst || src == dst) return CP_ERR_INVALID_ARG;
  const bool thd = desc->cu_seqlens_host != nullptr;
  if (thd && !desc->cu_seqlens_dev) return CP_ERR_INVALID_ARG;
  ProfScope ps(CP_K_ROPE, static_cast<cudaStream_t>(stream));
  return launch_permute_rope(idx, thd ? desc->cu_seqlens_dev : nullptr, thd ? desc->n_seqs : 0, desc->batch,
                             desc->seqlen, heads, desc->head_dim, double(rope_base), src, dst, inverse != 0,
                             desc->dtype, static_cast<cudaStream_t>(stream));
}

cp_status cp_tile_attn_fwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           int64_t q_row0, int64_t q_pos0, int64_t q_len, int64_t kv_row0,
                           int64_t kv_pos0, int64_t kv_len, float* o_part, float* lse_part,
                           void* stream) {
  cp_status st = validate_shape(desc);  // one edge needs no split rule
  if (st != CP_OK) return st;
  st = attn_kernels_for(*desc);
  if (st != CP_OK) return st;
  if (q_len < 0 || kv_len < 0 || q_row0 < 0 || kv_row0 < 0) return CP_ERR_INVALID_ARG;
  if (q_row0 + q_len > desc->seqlen || kv_row0 + kv_len > desc->seqlen) return CP_ERR_INVALID_ARG;
  if (std::llabs(q_pos0) >= (int64_t(1) << 30) || std::llabs(kv_pos0) >= (int64_t(1) << 30))
    return CP_ERR_INVALID_ARG;
  if (q_len == 0) return CP_OK;
  if (!q || !k || !v || !o_part || !lse_part) return CP_ERR_INVALID_ARG;
  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.o_out = nullptr;
  a.lse_out = nullptr;
  a.items = nullptr;
  a.segs = nullptr;
  a.edge = SingleEdge{int32_t(q_row0), int32_t(q_pos0), int32_t(q_len),
                      int32_t(kv_row0), int32_t(kv_pos0), int32_t(kv_len), desc->window};
  a.n_items = int32_t((q_len + kTile - 1) / kTile);
  a.wide_items = nullptr;
  a.wide_segs = nullptr;
  a.n_wide_items = int32_t((q_len + kWideRows - 1) / kWideRows);
  a.batch = desc->batch;
  a.H = desc->heads_q;
  a.Hkv = desc->heads_kv;
  a.d = desc->head_dim;
  a.seqlen = desc->seqlen;
  a.part_rows = q_len;
  a.scale = eff_scale(*desc);
  a.causal = desc->causal;
  a.dtype = desc->dtype;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(CP_K_TILE_FWD, s);
  return a.dtype == CP_BF16 ? launch_fwd_tc(a, s) : launch_fwd_simt(a, s);
}

cp_status cp_merge_partials(int32_t n_parts, int64_t rows, int32_t heads, int32_t head_dim,
                            const float* o_parts, const float* lse_parts, void* o_out,
                            cp_dtype out_dtype, float* lse_out, void* stream) {
  if (n_parts < 1 || rows < 0 || heads < 1) return CP_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return CP_ERR_UNSUPPORTED;
  if (out_dtype != CP_F32 && out_dtype != CP_BF16) return CP_ERR_UNSUPPORTED;
  if (rows >= (int64_t(1) << 31) || int64_t(n_parts) * rows >= (int64_t(1) << 31))
    return CP_ERR_UNSUPPORTED;
  if (rows == 0) return CP_OK;
  if (!o_parts || !lse_parts || !o_out) return CP_ERR_INVALID_ARG;
  MergeArgs a{};
  a.o_part = o_parts;
  a.lse_part = lse_parts;
  a.o_out = o_out;
  a.lse_out = lse_out;
  a.segs = nullptr;
  a.dense = MergeSeg{0, int32_t(rows), 0, n_parts, int32_t(rows), 0, {0, 0}};
  a.n_segs = 1;
  a.merge_rows = rows;
  a.batch = 1;
  a.H = heads;
  a.d = head_dim;
  a.part_rows = int64_t(n_parts) * rows;
  a.out_rows = rows;
  a.out_dtype = out_dtype;
  ProfScope ps(CP_K_MERGE, static_cast<cudaStream_t>(stream));
  return launch_merge(a, static_cast<cudaStream_t>(stream));
}

cp_status cp_ring_attn_fwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  cp_status st;
  if (!desc) return CP_ERR_INVALID_ARG;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  st = attn_kernels_for(*desc);
  if (st != CP_OK) return st;
  if (desc->seqlen == 0) return CP_OK;
  if (!q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(*desc, *p, false);
  if (!ws || !aligned256(ws)) return CP_ERR_INVALID_ARG;
  if (ws_bytes < w.total) return CP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  st = upload(base + w.tables, p->fwd_image, &p->fwd_pinned, s);
  if (st != CP_OK) return st;
  unsigned char* tables = base + w.tables;

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
  a.scale = eff_scale(*desc);
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

cp_status cp_ring_attn_bwd(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* ws, size_t ws_bytes, void* stream) {
  cp_status st;
  if (!desc) return CP_ERR_INVALID_ARG;
  auto p = get_plan(*desc, &st);
  if (!p) return st;
  st = attn_kernels_for(*desc);
  if (st != CP_OK) return st;
  if (desc->seqlen == 0) return CP_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return CP_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(*desc, *p, true);
  if (!ws || !aligned256(ws)) return CP_ERR_INVALID_ARG;
  if (ws_bytes < w.total) return CP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(ws);
  st = upload(base + w.tables, p->bwd_image, &p->bwd_pinned, s);
  if (st != CP_OK) return st;
  unsigned char* tables = base + w.tables;

  BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.lse = lse;
  a.delta = reinterpret_cast<float*>(base + w.delta);
  a.lse2 = reinterpret_cast<float*>(base + w.lse2);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = w.dq_acc ? reinterpret_cast<float*>(base + w.dq_acc) : nullptr;
  a.kv_items = reinterpret_cast<const TileItem*>(tables + p->off_kv_items);
  a.kv_segs = reinterpret_cast<const Seg*>(tables + p->off_kv_segs);
  a.n_kv_items = int32_t(p->kv_items.size());
  a.kv_work = reinterpret_cast<const int32_t*>(tables + p->off_kv_work);
  a.kv_cta = reinterpret_cast<const int32_t*>(tables + p->off_kv_cta);
  a.kv_grid = p->kv_grid;
  a.q_items = reinterpret_cast<const TileItem*>(tables + p->off_q_items);
  a.q_segs = reinterpret_cast<const Seg*>(tables + p->off_q_segs);
  a.n_q_items = int32_t(p->q_items.size());
  a.batch = desc->batch;
  a.H = desc->heads_q;
  a.Hkv = desc->heads_kv;
  a.d = desc->head_dim;
  a.seqlen = desc->seqlen;
  a.scale = eff_scale(*desc);
  a.causal = desc->causal;
  a.dtype = desc->dtype;

  const bool tc = a.dtype == CP_BF16;
  if (tc && !a.dq_acc) return CP_ERR_INVALID_ARG;  // the layout reserves the accumulator for every bf16 call
  {
    ProfScope ps(CP_K_DELTA, s);
    st = launch_bwd_prep(o, dout, lse, const_cast<float*>(a.delta), const_cast<float*>(a.lse2),
                         a.batch, a.seqlen, a.H, a.d, a.dtype, tc ? a.dq_acc : nullptr,
                         tc ? int64_t(dq_acc_floats(*desc)) : 0, s);
  }
  if (st != CP_OK) return st;
  if (!tc) {
    ProfScope ps(CP_K_TILE_BWD, s, 2);
    return launch_bwd_simt(a, s);
  }
  {
    ProfScope ps(CP_K_TILE_BWD, s);
    st = launch_bwd_tc(a, s);
  }
  if (st != CP_OK) return st;
  ProfScope ps(CP_K_CONVERT, s);
  return launch_dq_post(a, s);
}

cp_status cp_debug_set_wait_limit(int64_t cycles) { return set_wait_limit_cycles(cycles); }

cp_status cp_get_device_error(void* stream) {
  return read_and_clear_device_error(static_cast<cudaStream_t>(stream));
}

cp_status cp_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
  return CP_OK;
}

cp_status cp_profile_read(double* ms, int64_t* launches) {
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    recs.swap(g_prof_recs);
    if (launches)
      for (int i = 0; i < CP_K_COUNT; ++i) launches[i] = g_prof_launches[i];
    for (int i = 0; i < CP_K_COUNT; ++i) g_prof_launches[i] = 0;
  }
  if (ms)
    for (int i = 0; i < CP_K_COUNT; ++i) ms[i] = 0.0;
  cp_status st = CP_OK;
  for (const ProfRecord& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      st = CP_ERR_CUDA;
    else if (ms)
      ms[r.kid] += t;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (const ProfRecord& r : recs) {
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  return st;
}

}  // extern "C"
