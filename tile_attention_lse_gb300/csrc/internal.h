// Shared host/device definitions of libcpattn: the task-graph tables that the
// host planner writes and the kernels read, and the launch entry points of
// every kernel translation unit.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "cpattn.h"

namespace cpattn {

// Stationary tile height (queries in the forward pass, keys in the backward)
// and streamed tile width.  128 is the M of one tcgen05.mma (cta_group::1).
constexpr int kTile = 128;
// Query rows of one tensor-core forward item: two stationary Q tiles that
// share each streamed K/V tile.
constexpr int kWideRows = 2 * kTile;
// Streamed key tiles per forward part: a Q tile's edges are walked in groups
// of about this many key tiles, each group emitting one partial state.
constexpr int kPartTiles = 128;

// A run of consecutive tokens: `len` rows starting at tensor row `row0`
// (within one batch entry), holding positions pos0 .. pos0+len-1 of one
// (sub-)sequence.  win > 0 bounds the band of the sliding-window mask between
// this segment and the stationary tile it is streamed against: key position
// kp and query position qp see each other iff kp <= qp (causal) and
// qp - kp < win; win = 0 leaves the band open.
struct Seg {
  int32_t row0;
  int32_t pos0;
  int32_t len;
  int32_t win;
};

// One unit of work: a stationary tile (<= kTile rows) and the list of
// segments streamed against it.
//  forward:            stationary = Q tile, segments = the K/V chunks of one
//                      streaming part (consecutive task-graph edges in ring
//                      order, ordered by position), out_row0 = partial row,
//                      or -1 when the part is the Q chunk's only one: the
//                      item then writes the final O and LSE of its own rows
//  backward dK/dV:     stationary = K/V tile, segments = every Q range that
//                      sees it (all query ranks, ring order)
//  backward dQ (SIMT): stationary = Q tile, segments = every visible K/V range
struct TileItem {
  int32_t row0;
  int32_t pos0;
  int32_t len;
  int32_t seg_begin;
  int32_t seg_count;
  int32_t out_row0;
  int32_t cost;  // streamed kTile x kTile tiles (host-side ordering key)
  int32_t pad;
};

// Merge of the partial states of one Q chunk: partial e of local row i sits at
// partial row part_row0 + e * part_stride + i; output row out_row0 + i.
struct MergeSeg {
  int32_t out_row0;
  int32_t len;
  int32_t part_row0;
  int32_t n_parts;
  int32_t part_stride;
  int32_t merge_row0;  // first merge row of this segment (prefix sum of len)
  int32_t pad[2];
};

// Single-edge mode (cp_tile_attn_fwd): no tables, the items are the 128-row
// (SIMT) or kWideRows-row (tensor core) tiles of one query range against one
// key range.
struct SingleEdge {
  int32_t q_row0, q_pos0, q_len;
  int32_t kv_row0, kv_pos0, kv_len;
  int32_t win;  // sliding-window band (0: none)
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  float* o_part;    // [batch][part_rows][H][d]
  float* lse_part;  // [batch][part_rows][H]
  // outputs (layout of q; lse [batch][seqlen][H], natural log) for the
  // items with out_row0 = -1 (single-part Q chunks); null in single-edge mode
  void* o_out;
  float* lse_out;
  const TileItem* items;  // 128-row items, one per (Q tile, streaming part); nullptr -> single-edge mode
  const Seg* segs;
  const TileItem* wide_items;  // kWideRows-row items of the same parts (tensor-core path)
  const Seg* wide_segs;
  int32_t n_wide_items;
  SingleEdge edge;
  int32_t n_items;
  int32_t batch, H, Hkv, d;
  int64_t seqlen;     // rows per batch entry of q/k/v
  int64_t part_rows;  // partial rows per batch entry
  float scale;
  int32_t causal;
  cp_dtype dtype;
};

struct MergeArgs {
  const float* o_part;
  const float* lse_part;
  void* o_out;
  float* lse_out;
  const MergeSeg* segs;  // nullptr -> dense mode using `dense`
  MergeSeg dense;
  int32_t n_segs;
  int64_t merge_rows;  // rows per batch entry covered by the segments
  int32_t batch, H, d;
  int64_t part_rows;   // partial rows per batch entry
  int64_t out_rows;    // output rows per batch entry
  cp_dtype out_dtype;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* lse;    // [batch][seqlen][H], natural log
  const float* delta;  // [batch][H][seqlen]: D = <dO, O>
  const float* lse2;   // [batch][H][seqlen]: lse * log2(e), +inf for an empty row
  void* dq;
  void* dk;
  void* dv;
  // float32 dQ accumulator of the tensor-core path (zeroed by the backward
  // preprocess): [batch * q-heads][seqlen][128].  Null elsewhere.
  float* dq_acc;
  const TileItem* kv_items;
  const Seg* kv_segs;
  int32_t n_kv_items;
  // tensor-core schedule: CTA c runs work indices kv_work[kv_cta[c] ..
  // kv_cta[c + 1]) on a grid of kv_grid CTAs
  const int32_t* kv_work;
  const int32_t* kv_cta;
  int32_t kv_grid;
  const TileItem* q_items;
  const Seg* q_segs;
  int32_t n_q_items;
  int32_t batch, H, Hkv, d;
  int64_t seqlen;
  float scale;
  int32_t causal;
  cp_dtype dtype;
};

// ---- launchers (each returns CP_OK or CP_ERR_CUDA / CP_ERR_UNSUPPORTED) ----
cp_status launch_partition(int32_t cp, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                           int32_t* idx, int32_t* local_cu, int striped, cudaStream_t s);
cp_status launch_partition_hybrid(int32_t cp, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                                  const int32_t* gcp_dev, const int32_t* g0_dev, int32_t* idx, int32_t* local_cu,
                                  cudaStream_t s);
cp_status launch_token_seq_pos(const int32_t* idx, int64_t seqlen, const int32_t* cu_dev, int32_t n_seqs,
                               int32_t* seq_pos, cudaStream_t s);
cp_status launch_permute(const int32_t* idx, int32_t batch, int64_t seqlen, int64_t row_bytes,
                         const void* src, void* dst, int inverse, cudaStream_t s);
// Token gather with rotary position embedding (cu_dev null for BSHD).
cp_status launch_permute_rope(const int32_t* idx, const int32_t* cu_dev, int32_t n_seqs, int32_t batch,
                              int64_t seqlen, int32_t heads, int32_t d, double base, const void* src, void* dst,
                              int inverse, cp_dtype dtype, cudaStream_t s);
cp_status launch_fwd_simt(const FwdArgs& a, cudaStream_t s);
cp_status launch_fwd_tc(const FwdArgs& a, cudaStream_t s);
// The tcgen05 kernels can run here: the driver exports the tensor-map encoder.
bool tc_available();
cp_status launch_merge(const MergeArgs& a, cudaStream_t s);
// Also zeroes `zero_floats` floats at `zero` (a multiple of 4, 16-byte
// aligned; null for none).
cp_status launch_bwd_prep(const void* o, const void* dout, const float* lse, float* delta,
                          float* lse2, int32_t batch, int64_t S, int32_t H, int32_t d,
                          cp_dtype dtype, float* zero, int64_t zero_floats, cudaStream_t s);
cp_status launch_bwd_simt(const BwdArgs& a, cudaStream_t s);
cp_status launch_bwd_tc(const BwdArgs& a, cudaStream_t s);
// dQ = scale * the tensor-core path's float32 accumulator, as bf16.
cp_status launch_dq_post(const BwdArgs& a, cudaStream_t s);
// Copies `bytes` (a multiple of 16, both pointers 16-byte aligned) from
// device-mapped pinned host memory with the GPU's own loads, so the copy
// never waits behind the caller's transfers on a copy engine.
cp_status launch_copy_from_host(void* dst, const void* src_mapped, size_t bytes, cudaStream_t s);

// Device error word (set by bounded waits that ran out).
cp_status read_and_clear_device_error(cudaStream_t s);

inline cp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CP_OK : CP_ERR_CUDA; }

// Benchmark instrumentation (cp_profile_enable): counts the launches of one
// kernel class and, with timing on, brackets them with two CUDA events on the
// stream they run on.
class ProfScope {
 public:
  ProfScope(int kernel_class, cudaStream_t s, int n_launches = 1);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  int kid_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace cpattn

namespace cpattn {
// Device address of the library's error word on the current device.
int* device_error_ptr();
// Cycle budget of the tensor-core kernels' main-loop waits: the default of
// about two seconds unless cp_debug_set_wait_limit set another.
long long wait_limit_cycles();
// cycles <= 0 restores the default; above the default: CP_ERR_INVALID_ARG.
cp_status set_wait_limit_cycles(int64_t cycles);
}  // namespace cpattn
