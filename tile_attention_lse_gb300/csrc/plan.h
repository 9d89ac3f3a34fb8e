// Host planner: turns a descriptor into the task graph of the ring walk.
#pragma once

#include <memory>
#include <vector>

#include "internal.h"

namespace cpattn {

struct Plan {
  // forward: one item per (Q tile, key owner) edge, heaviest first
  std::vector<TileItem> fwd_items;
  std::vector<Seg> fwd_segs;
  // the same edges cut into kWideRows-row query tiles (tensor-core forward:
  // two 128-row Q tiles share every K/V tile), heaviest first
  std::vector<TileItem> fwd_wide;
  std::vector<Seg> fwd_wide_segs;
  std::vector<MergeSeg> merge_segs;
  // backward: K/V-stationary items (dK, dV; dQ by accumulation) and
  // Q-stationary items (dQ of the SIMT path)
  std::vector<TileItem> kv_items;
  std::vector<Seg> kv_segs;
  std::vector<TileItem> q_items;
  std::vector<Seg> q_segs;
  // tensor-core backward schedule: work index w = (batch * kv-head) *
  // kv_items.size() + item, per CTA in kv_cta[c] .. kv_cta[c + 1] of kv_work,
  // in increasing w (head-major), each item given to the least-loaded CTA so
  // the CTAs move through the heads together (one head's Q, dO, K, V and dQ
  // accumulator stay in L2)
  std::vector<int32_t> kv_work;
  std::vector<int32_t> kv_cta;
  int32_t kv_grid = 0;

  int64_t part_rows = 0;     // partial rows per batch entry
  int64_t merge_rows = 0;    // rows covered by merge_segs per batch entry
  int64_t pairs = 0;         // unmasked (query, key) pairs per batch entry and head
  int64_t fwd_tiles = 0;     // streamed key tiles over all forward items

  // Byte offsets of each table inside the packed table image.
  size_t off_fwd_items = 0, off_fwd_segs = 0, off_merge = 0;
  size_t off_fwd_wide = 0, off_fwd_wide_segs = 0;
  size_t off_kv_items = 0, off_kv_segs = 0, off_q_items = 0, off_q_segs = 0;
  size_t off_kv_work = 0, off_kv_cta = 0;
  size_t fwd_table_bytes = 0;  // [0, fwd_table_bytes): forward tables
  size_t bwd_table_bytes = 0;  // backward tables image size
  std::vector<unsigned char> fwd_image, bwd_image;
  void* fwd_pinned = nullptr;  // pinned copies used as async upload sources
  void* bwd_pinned = nullptr;
  ~Plan();
};

// Builds (or returns the cached) plan; nullptr if the descriptor is invalid.
std::shared_ptr<Plan> get_plan(const cp_attn_desc& d, cp_status* st);

// Workspace layout.
struct WsLayout {
  size_t tables = 0;     // offset of the table image
  size_t part_o = 0, part_l = 0;  // forward
  size_t delta = 0, lse2 = 0;   // backward
  size_t dq_acc = 0;            // backward, bf16 head_dim 128: float32 dQ accumulator (0 = none)
  size_t total = 0;
};
WsLayout ws_layout(const cp_attn_desc& d, const Plan& p, bool backward);
// Floats of the tensor-core backward's float32 dQ accumulator (layout in BwdArgs).
size_t dq_acc_floats(const cp_attn_desc& d);

// Shapes, types and sizes only.
cp_status validate_shape(const cp_attn_desc* d);
// validate_shape plus the split rules (cu_seqlens, lengths % 2*cp).
cp_status validate(const cp_attn_desc* d);

}  // namespace cpattn
