// Host planner of the Q-KV task graph ("Context Parallelism (CP)" §2.1,
// edge set of the causal bipartite graph; §2.3 strategy 1, Q stays and K/V
// moves around the ring) for the zigzag / per-sub-sequence split
// ("04 · Megatron-LM 实现" §1.1, §1.2).
//
// Chunks: every (sub-)sequence k of length len_k is cut into 2*cp chunks of
// c_k = len_k / (2*cp) tokens; chunk a belongs to rank a (a < cp) or
// 2*cp-1-a.  Rank r at ring step t holds the K/V of owner s = (r - t) mod cp
// ("Sequence Parallelism + Ring Attention" §2: step 0 is the local block, then
// the block of the previous card).  The edge (Q chunk a, owner s) exists when
// some query of a sees some key of chunks {s, 2cp-1-s}: causally iff s <= a.
// Consecutive edges of a Q chunk are walked as streaming parts; a chunk of
// two or more parts gets one partial state per part (laid out part after
// part, in ring-step order) and a merge segment, a chunk of one part is
// written to the outputs directly by its items.
#include "plan.h"

#include "tmap.h"

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <queue>
#include <string>
#include <utility>
#include <vector>

namespace cpattn {

Plan::~Plan() {
  if (fwd_pinned) cudaFreeHost(fwd_pinned);
  if (bwd_pinned) cudaFreeHost(bwd_pinned);
}

cp_status validate_shape(const cp_attn_desc* d) {
  if (!d) return CP_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads_q < 1 || d->heads_kv < 1 || d->cp < 1 || d->seqlen < 0)
    return CP_ERR_INVALID_ARG;
  if (d->dtype != CP_F32 && d->dtype != CP_BF16) return CP_ERR_UNSUPPORTED;
  if (d->order != CP_ORDER_ORIGINAL && d->order != CP_ORDER_RANK_LOCAL) return CP_ERR_INVALID_ARG;
  if (d->heads_q % d->heads_kv != 0) return CP_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return CP_ERR_UNSUPPORTED;
  if (d->seqlen >= (int64_t(1) << 30)) return CP_ERR_UNSUPPORTED;
  // token rows are 32-bit TMA coordinates and kernel row indices
  if (int64_t(d->batch) * d->seqlen >= (int64_t(1) << 31)) return CP_ERR_UNSUPPORTED;
  if (!(d->softmax_scale >= 0.0f)) return CP_ERR_INVALID_ARG;
  if (d->partition != CP_PARTITION_ZIGZAG && d->partition != CP_PARTITION_STRIPED) return CP_ERR_INVALID_ARG;
  // striped: a rank's tokens are strided in the original order, so the ring
  // walks rank-local tensors only
  if (d->partition == CP_PARTITION_STRIPED && d->order != CP_ORDER_RANK_LOCAL) return CP_ERR_UNSUPPORTED;
  if (d->window < 0 || d->window >= (1 << 30)) return CP_ERR_INVALID_ARG;
  if (d->window > 0 && !d->causal) return CP_ERR_UNSUPPORTED;  // a causal band only
  return CP_OK;
}

cp_status validate(const cp_attn_desc* d) {
  const cp_status st = validate_shape(d);
  if (st != CP_OK) return st;
  const int64_t align = (d->partition == CP_PARTITION_STRIPED ? 1 : 2) * int64_t(d->cp);
  const bool hybrid = d->seq_cp_host != nullptr;
  if (hybrid && (!d->cu_seqlens_host || !d->seq_rank0_host || d->partition != CP_PARTITION_ZIGZAG))
    return CP_ERR_INVALID_ARG;
  if (d->cu_seqlens_host) {
    if (d->batch != 1 || d->n_seqs < 0) return CP_ERR_INVALID_ARG;
    const int32_t* cu = d->cu_seqlens_host;
    if (cu[0] != 0 || cu[d->n_seqs] != d->seqlen) return CP_ERR_INVALID_ARG;
    for (int i = 0; i < d->n_seqs; ++i) {
      const int64_t len = int64_t(cu[i + 1]) - cu[i];
      if (len < 0) return CP_ERR_INVALID_ARG;
      if (hybrid) {  // an aligned power-of-two group of ranks per sub-sequence
        const int32_t g = d->seq_cp_host[i], r0 = d->seq_rank0_host[i];
        if (g < 1 || (g & (g - 1)) || g > d->cp || r0 < 0 || r0 % g || r0 + g > d->cp) return CP_ERR_INVALID_ARG;
        if (len % (2 * int64_t(g)) != 0) return CP_ERR_ALIGNMENT;
      } else if (len % align != 0) {
        return CP_ERR_ALIGNMENT;
      }
    }
  } else {
    if (d->n_seqs != 0 && d->n_seqs != 1) return CP_ERR_INVALID_ARG;
    if (d->seqlen % align != 0) return CP_ERR_ALIGNMENT;
  }
  return CP_OK;
}

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int owner(int a, int cp) { return a < cp ? a : 2 * cp - 1 - a; }

int32_t tiles_of(int64_t n) { return int32_t((n + kTile - 1) / kTile); }

// Offsets [lo, hi) of the keys of `kv` that some query at positions
// qfirst .. qlast can see: causally kp <= qlast, and inside the sliding-window
// band qfirst - kp < kv.win.  Empty when lo == hi.
std::pair<int64_t, int64_t> key_range(const Seg& kv, int64_t qfirst, int64_t qlast, bool causal) {
  int64_t hi = kv.len, lo = 0;
  if (causal) hi = std::min<int64_t>(hi, qlast - kv.pos0 + 1);
  if (kv.win > 0) lo = std::max<int64_t>(0, qfirst - kv.win + 1 - kv.pos0);
  return {lo, std::max(lo, hi)};
}

// Offsets [lo, hi) of the queries of `q` that see some key at positions
// kfirst .. klast (the same two bounds seen from the other side).
std::pair<int64_t, int64_t> query_range(const Seg& q, int64_t kfirst, int64_t klast, bool causal) {
  int64_t lo = causal ? std::max<int64_t>(0, kfirst - q.pos0) : 0, hi = q.len;
  if (q.win > 0) hi = std::min<int64_t>(hi, klast + q.win - q.pos0);
  return {lo, std::max(lo, hi)};
}

Seg sub_seg(const Seg& sg, int64_t lo, int64_t hi) {
  return Seg{int32_t(sg.row0 + lo), int32_t(sg.pos0 + lo), int32_t(hi - lo), sg.win};
}

// Causal pairs of a sequence of n tokens under a window of w (0: none).
int64_t band_pairs(int64_t n, int64_t w) {
  if (w <= 0 || w >= n) return n * (n + 1) / 2;
  return w * (w + 1) / 2 + (n - w) * w;
}

template <class T>
void append_bytes(std::vector<unsigned char>& img, size_t& off, const std::vector<T>& v) {
  off = align_up(img.size(), 256);
  img.resize(off + v.size() * sizeof(T));
  if (!v.empty()) std::memcpy(img.data() + off, v.data(), v.size() * sizeof(T));
}

void build(const cp_attn_desc& d, Plan& p) {
  const int cp = d.cp;
  const bool causal = d.causal != 0;
  std::vector<int64_t> cu;
  if (d.cu_seqlens_host) {
    for (int i = 0; i <= d.n_seqs; ++i) cu.push_back(d.cu_seqlens_host[i]);
  } else {
    cu = {0, d.seqlen};
  }
  const int64_t per_rank = d.seqlen / cp;
  // Hybrid CP: sub-sequence k on ranks g0[k] .. g0[k] + gcp[k] - 1 (else all
  // ranks); rank r's stream holds the slices of the sub-sequences whose group
  // contains r, in order, and the streams follow each other rank by rank.
  const bool hybrid = d.seq_cp_host != nullptr;
  const size_t nseq = cu.size() - 1;
  std::vector<int32_t> gcp(nseq, cp), g0(nseq, 0);
  std::vector<int64_t> slice0;  // [cp][nseq]: first row of rank r's slice of k
  if (hybrid) {
    for (size_t k = 0; k < nseq; ++k) {
      gcp[k] = d.seq_cp_host[k];
      g0[k] = d.seq_rank0_host[k];
    }
    slice0.assign(size_t(cp) * nseq, 0);
    int64_t row = 0;
    for (int r = 0; r < cp; ++r)
      for (size_t k = 0; k < nseq; ++k) {
        slice0[size_t(r) * nseq + k] = row;
        if (r >= g0[k] && r < g0[k] + gcp[k]) row += (cu[k + 1] - cu[k]) / gcp[k];
      }
  }
  // chunk a of 2 gcp[k] chunks of sub-sequence k (chunk length c)
  auto chunk_row = [&](size_t k, int a, int64_t c) -> int64_t {
    if (d.order == CP_ORDER_ORIGINAL) return cu[k] + int64_t(a) * c;
    const int g = gcp[k];
    const int r = owner(a, g);
    const int64_t base = hybrid ? slice0[size_t(g0[k] + r) * nseq + k] : int64_t(r) * per_rank + cu[k] / cp;
    return base + (a < g ? 0 : c);
  };

  const bool striped = d.partition == CP_PARTITION_STRIPED;
  const int64_t win = d.window;
  // Striped: the window between query rank r and key rank s in the ranks'
  // own slot numbers (query slot w, key slot u at virtual position u + d,
  // d = [s > r]).  Token distance (r + cp w) - (s + cp u) < W iff w - u <
  // M = ceil((W + s - r) / cp), i.e. qv - kv < M - d.  0 when no pair of the
  // two ranks is in the band (the edge is dropped), -1 without a window.
  auto striped_win = [&](int r, int s_) -> int64_t {
    if (win == 0) return -1;
    const int64_t x = win + s_ - r;
    if (x <= 0) return 0;
    return std::max<int64_t>(0, (x + cp - 1) / cp - (s_ > r ? 1 : 0));
  };
  // first row of rank r's stream of sub-sequence k (rank-local order)
  auto rank_row = [&](size_t k, int r) -> int64_t { return int64_t(r) * per_rank + cu[k] / cp; };

  for (size_t k = 0; k + 1 < cu.size(); ++k) {
    const int64_t len = cu[k + 1] - cu[k];
    if (len == 0) continue;
    p.pairs += causal ? band_pairs(len, win) : len * len;

    // Query chunks of this sequence, each with its edges in ring order (key
    // owner s = (r - t) mod cp, t = 0 .. cp-1).
    //  zigzag: chunk a of 2cp (length c = len / 2cp) on rank owner(a); an
    //    edge is the owner's chunks s and 2cp-1-s that the chunk can see.
    //  striped: rank r's stream (len / cp tokens, token r + cp u at local row
    //    u) against rank s's stream.  Positions are virtual: the local row.
    //    Key u of rank s is visible to query w of rank r iff s + cp u <=
    //    r + cp w, i.e. u + [s > r] <= w, so rank s's keys start at virtual
    //    position [s > r] and the tile kernels' position masks apply as is.
    struct QChunk {
      int64_t row, pos, len;
      std::vector<std::vector<Seg>> edges;
    };
    std::vector<QChunk> qchunks;
    if (!striped) {
      // the ring of this sub-sequence's group (hybrid CP), else of all ranks
      const int g = gcp[k];
      const int64_t c = len / (2 * g);
      for (int a = 0; a < 2 * g; ++a) {
        QChunk q{chunk_row(k, a, c), int64_t(a) * c, c, {}};
        const int r = owner(a, g);
        for (int t = 0; t < g; ++t) {
          const int s_ = ((r - t) % g + g) % g;
          std::vector<Seg> segs;
          for (int b : {s_, 2 * g - 1 - s_}) {
            const Seg sg{int32_t(chunk_row(k, b, c)), int32_t(int64_t(b) * c), int32_t(c), int32_t(win)};
            const auto rg = key_range(sg, q.pos, q.pos + c - 1, causal);
            if (rg.second > rg.first) segs.push_back(sg);
          }
          if (!segs.empty()) q.edges.push_back(segs);
        }
        qchunks.push_back(std::move(q));
      }
    } else {
      const int64_t cl = len / cp;
      for (int r = 0; r < cp; ++r) {
        QChunk q{rank_row(k, r), 0, cl, {}};
        for (int t = 0; t < cp; ++t) {
          const int s_ = ((r - t) % cp + cp) % cp;
          const int64_t w = striped_win(r, s_);
          if (w == 0) continue;
          const Seg sg{int32_t(rank_row(k, s_)), int32_t(s_ > r ? 1 : 0), int32_t(cl), int32_t(std::max<int64_t>(w, 0))};
          const auto rg = key_range(sg, 0, cl - 1, causal);
          if (rg.second > rg.first) q.edges.push_back({sg});
        }
        qchunks.push_back(std::move(q));
      }
    }

    // Streaming parts of a Q chunk: consecutive edges grouped into parts of
    // about kPartTiles streamed key tiles.  One part is walked with one
    // online (m, l, acc) state and emits one partial state, merged by the LSE
    // merge; inside a part the segments are ordered by position (zigzag: the
    // diagonal chunk, in the owner's own edge, ends the first part, so a Q
    // tile's visible keys form a prefix).
    auto parts_of = [&](const QChunk& q) {
      const int64_t qlast = q.pos + q.len - 1;
      std::vector<int64_t> edge_tiles;
      for (const auto& e : q.edges) {
        int64_t tl = 0;
        for (const Seg& sg : e) {
          const auto rg = key_range(sg, q.pos, qlast, causal);
          tl += tiles_of(rg.second - rg.first);
        }
        edge_tiles.push_back(tl);
      }
      int64_t total = 0;
      for (int64_t x : edge_tiles) total += x;
      const int64_t want = std::max<int64_t>(1, std::min<int64_t>(int64_t(q.edges.size()),
                                                                  (total + kPartTiles - 1) / kPartTiles));
      std::vector<std::vector<Seg>> parts(1);
      int64_t acc = 0;
      for (size_t e = 0; e < q.edges.size(); ++e) {
        // start a new part once this one holds its share of the tiles
        if (!parts.back().empty() && int64_t(parts.size()) < want &&
            acc * want >= total * int64_t(parts.size()))
          parts.emplace_back();
        parts.back().insert(parts.back().end(), q.edges[e].begin(), q.edges[e].end());
        acc += edge_tiles[e];
      }
      for (auto& part : parts)
        std::stable_sort(part.begin(), part.end(), [](const Seg& x, const Seg& y) { return x.pos0 < y.pos0; });
      return parts;
    };

    std::vector<std::vector<std::vector<Seg>>> all_parts;
    for (const QChunk& q : qchunks) all_parts.push_back(parts_of(q));
    std::vector<int64_t> part0_of(qchunks.size(), 0);  // first partial row of each Q chunk

    // ---- forward items and merge segments, per Q chunk ----
    for (size_t qi = 0; qi < qchunks.size(); ++qi) {
      const QChunk& q = qchunks[qi];
      const auto& parts = all_parts[qi];
      const int64_t qrow = q.row, qpos = q.pos, c = q.len;
      // A Q chunk walked in one part needs no merge: its items write the
      // final O and LSE into the output rows themselves (out_row0 = -1).
      // Only chunks of two or more parts get partial rows and a merge segment.
      const bool direct = parts.size() == 1;
      const int64_t part0 = direct ? -1 : p.part_rows;
      part0_of[qi] = part0;
      if (!direct) {
        p.merge_segs.push_back(MergeSeg{int32_t(qrow), int32_t(c), int32_t(part0),
                                        int32_t(parts.size()), int32_t(c), int32_t(p.merge_rows), {0, 0}});
        p.merge_rows += c;
        p.part_rows += int64_t(parts.size()) * c;
      }
      for (int64_t t0 = 0; t0 < c; t0 += kTile) {
        const int64_t tl = std::min<int64_t>(kTile, c - t0);
        const int64_t qlast = qpos + t0 + tl - 1;
        std::vector<Seg> all;  // every visible segment of this Q tile (dQ item)
        for (size_t e = 0; e < parts.size(); ++e) {
          TileItem it{};
          it.row0 = int32_t(qrow + t0);
          it.pos0 = int32_t(qpos + t0);
          it.len = int32_t(tl);
          it.seg_begin = int32_t(p.fwd_segs.size());
          it.out_row0 = direct ? -1 : int32_t(part0 + int64_t(e) * c + t0);
          int32_t cost = 0;
          for (const Seg& sg : parts[e]) {
            const auto rg = key_range(sg, qpos + t0, qlast, causal);
            if (rg.second == rg.first) continue;
            const Seg ts = sub_seg(sg, rg.first, rg.second);
            p.fwd_segs.push_back(ts);
            all.push_back(ts);
            cost += tiles_of(ts.len);
          }
          it.seg_count = int32_t(p.fwd_segs.size()) - it.seg_begin;
          it.cost = cost;
          p.fwd_tiles += cost;
          p.fwd_items.push_back(it);
        }
        TileItem qi_{};
        qi_.row0 = int32_t(qrow + t0);
        qi_.pos0 = int32_t(qpos + t0);
        qi_.len = int32_t(tl);
        qi_.seg_begin = int32_t(p.q_segs.size());
        qi_.seg_count = int32_t(all.size());
        int32_t cost = 0;
        for (const Seg& sg : all) cost += tiles_of(sg.len);
        qi_.cost = cost;
        p.q_segs.insert(p.q_segs.end(), all.begin(), all.end());
        p.q_items.push_back(qi_);
      }
    }

    // ---- the same parts in kWideRows-row query tiles (tensor-core forward) ----
    for (size_t qi = 0; qi < qchunks.size(); ++qi) {
      const QChunk& q = qchunks[qi];
      const auto& parts = all_parts[qi];
      const int64_t qrow = q.row, qpos = q.pos, c = q.len, part0 = part0_of[qi];
      for (size_t e = 0; e < parts.size(); ++e) {
        for (int64_t t0 = 0; t0 < c; t0 += kWideRows) {
          const int64_t tl = std::min<int64_t>(kWideRows, c - t0);
          const int64_t qlast = qpos + t0 + tl - 1;
          TileItem it{};
          it.row0 = int32_t(qrow + t0);
          it.pos0 = int32_t(qpos + t0);
          it.len = int32_t(tl);
          it.seg_begin = int32_t(p.fwd_wide_segs.size());
          it.out_row0 = part0 < 0 ? -1 : int32_t(part0 + int64_t(e) * c + t0);
          int32_t cost = 0;
          for (const Seg& sg : parts[e]) {
            const auto rg = key_range(sg, qpos + t0, qlast, causal);
            if (rg.second == rg.first) continue;
            const Seg ts = sub_seg(sg, rg.first, rg.second);
            p.fwd_wide_segs.push_back(ts);
            cost += tiles_of(ts.len);
          }
          it.seg_count = int32_t(p.fwd_wide_segs.size()) - it.seg_begin;
          it.cost = cost;
          p.fwd_wide.push_back(it);
        }
      }
    }

    // ---- backward: K/V-stationary items; Q ranges of every rank that sees
    //      the tile, in ring order starting at the owner ----
    if (!striped) {
      const int g = gcp[k];
      const int64_t c = len / (2 * g);
      for (int b = 0; b < 2 * g; ++b) {
        const int s_ = owner(b, g);
        const int64_t krow = chunk_row(k, b, c), kpos = int64_t(b) * c;
        for (int64_t u0 = 0; u0 < c; u0 += kTile) {
          const int64_t tl = std::min<int64_t>(kTile, c - u0);
          TileItem it{};
          it.row0 = int32_t(krow + u0);
          it.pos0 = int32_t(kpos + u0);
          it.len = int32_t(tl);
          it.seg_begin = int32_t(p.kv_segs.size());
          int32_t cost = 0;
          for (int t = 0; t < g; ++t) {
            const int r = (s_ + t) % g;
            for (int a : {r, 2 * g - 1 - r}) {
              const Seg q{int32_t(chunk_row(k, a, c)), int32_t(int64_t(a) * c), int32_t(c), int32_t(win)};
              // queries before the tile's first key, or past its band, see nothing
              const auto rg = query_range(q, kpos + u0, kpos + u0 + tl - 1, causal);
              if (rg.second == rg.first) continue;
              p.kv_segs.push_back(sub_seg(q, rg.first, rg.second));
              cost += tiles_of(rg.second - rg.first);
            }
          }
          it.seg_count = int32_t(p.kv_segs.size()) - it.seg_begin;
          it.cost = cost;
          p.kv_items.push_back(it);
        }
      }
    } else {
      // striped: key tile of rank s at virtual positions u0 ..; rank r's
      // queries at virtual position w - [s > r] (the same relation as above)
      const int64_t cl = len / cp;
      for (int s_ = 0; s_ < cp; ++s_) {
        const int64_t krow = rank_row(k, s_);
        for (int64_t u0 = 0; u0 < cl; u0 += kTile) {
          const int64_t tl = std::min<int64_t>(kTile, cl - u0);
          TileItem it{};
          it.row0 = int32_t(krow + u0);
          it.pos0 = int32_t(u0);
          it.len = int32_t(tl);
          it.seg_begin = int32_t(p.kv_segs.size());
          int32_t cost = 0;
          for (int t = 0; t < cp; ++t) {
            const int r = (s_ + t) % cp;
            const int64_t dv = s_ > r ? 1 : 0, w = striped_win(r, s_);
            if (w == 0) continue;
            const Seg q{int32_t(rank_row(k, r)), int32_t(-dv), int32_t(cl), int32_t(std::max<int64_t>(w, 0))};
            const auto rg = query_range(q, u0, u0 + tl - 1, causal);
            if (rg.second == rg.first) continue;
            p.kv_segs.push_back(sub_seg(q, rg.first, rg.second));
            cost += tiles_of(rg.second - rg.first);
          }
          it.seg_count = int32_t(p.kv_segs.size()) - it.seg_begin;
          it.cost = cost;
          p.kv_items.push_back(it);
        }
      }
    }
  }

  // Heaviest items first (longest-processing-time order for the persistent
  // kernels; ties keep plan order).
  auto heavier = [](const TileItem& x, const TileItem& y) { return x.cost > y.cost; };
  std::stable_sort(p.fwd_items.begin(), p.fwd_items.end(), heavier);
  std::stable_sort(p.fwd_wide.begin(), p.fwd_wide.end(), heavier);
  std::stable_sort(p.kv_items.begin(), p.kv_items.end(), heavier);
  std::stable_sort(p.q_items.begin(), p.q_items.end(), heavier);

  append_bytes(p.fwd_image, p.off_fwd_items, p.fwd_items);
  append_bytes(p.fwd_image, p.off_fwd_segs, p.fwd_segs);
  append_bytes(p.fwd_image, p.off_merge, p.merge_segs);
  append_bytes(p.fwd_image, p.off_fwd_wide, p.fwd_wide);
  append_bytes(p.fwd_image, p.off_fwd_wide_segs, p.fwd_wide_segs);
  p.fwd_image.resize(align_up(p.fwd_image.size(), 256));
  p.fwd_table_bytes = p.fwd_image.size();
  // Backward schedule (see Plan::kv_work): greedy least-loaded assignment in
  // head-major order; cost = streamed query tiles of the item + 1 (K/V load,
  // dK/dV epilogue).
  {
    const int64_t n_items = int64_t(p.kv_items.size());
    const int64_t n_bh = int64_t(d.batch) * d.heads_kv;
    const int64_t total = n_items * n_bh;
    const int group = d.heads_q / d.heads_kv;
    const int grid = int(std::min<int64_t>(total, num_sms()));
    p.kv_grid = grid;
    std::vector<std::vector<int32_t>> lists(size_t(std::max(grid, 0)));
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> least;
    for (int c = 0; c < grid; ++c) least.push(Load{0, c});
    for (int64_t w = 0; w < total && grid > 0; ++w) {
      const Load l = least.top();
      least.pop();
      lists[size_t(l.second)].push_back(int32_t(w));
      least.push(Load{l.first + int64_t(p.kv_items[size_t(w % n_items)].cost) * group + 1, l.second});
    }
    p.kv_cta.assign(1, 0);
    for (const auto& l : lists) {
      p.kv_work.insert(p.kv_work.end(), l.begin(), l.end());
      p.kv_cta.push_back(int32_t(p.kv_work.size()));
    }
  }
  append_bytes(p.bwd_image, p.off_kv_items, p.kv_items);
  append_bytes(p.bwd_image, p.off_kv_segs, p.kv_segs);
  append_bytes(p.bwd_image, p.off_q_items, p.q_items);
  append_bytes(p.bwd_image, p.off_q_segs, p.q_segs);
  append_bytes(p.bwd_image, p.off_kv_work, p.kv_work);
  append_bytes(p.bwd_image, p.off_kv_cta, p.kv_cta);
  p.bwd_image.resize(align_up(p.bwd_image.size(), 256));
  p.bwd_table_bytes = p.bwd_image.size();
}

std::string plan_key(const cp_attn_desc& d) {
  std::string key;
  auto put = [&](int64_t x) { key.append(reinterpret_cast<const char*>(&x), sizeof(x)); };
  put(d.cp);
  put(d.causal != 0);
  put(d.seqlen);
  put(d.batch);  // the backward schedule depends on batch and heads
  put(d.heads_q);
  put(d.heads_kv);
  put(d.order);
  put(d.partition);
  put(d.window);
  put(d.seq_cp_host ? 1 : 0);
  put(d.cu_seqlens_host ? d.n_seqs : -1);
  if (d.cu_seqlens_host)
    key.append(reinterpret_cast<const char*>(d.cu_seqlens_host), sizeof(int32_t) * (d.n_seqs + 1));
  if (d.seq_cp_host) {
    key.append(reinterpret_cast<const char*>(d.seq_cp_host), sizeof(int32_t) * d.n_seqs);
    key.append(reinterpret_cast<const char*>(d.seq_rank0_host), sizeof(int32_t) * d.n_seqs);
  }
  return key;
}

std::mutex g_mu;
std::map<std::string, std::shared_ptr<Plan>> g_cache;
constexpr size_t kMaxPlans = 32;

}  // namespace

std::shared_ptr<Plan> get_plan(const cp_attn_desc& d, cp_status* st) {
  *st = validate(&d);
  if (*st != CP_OK) return nullptr;
  const std::string key = plan_key(d);
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_cache.find(key);
  if (it != g_cache.end()) return it->second;
  auto p = std::make_shared<Plan>();
  build(d, *p);
  if (g_cache.size() >= kMaxPlans) g_cache.erase(g_cache.begin());
  g_cache[key] = p;
  return p;
}

size_t dq_acc_floats(const cp_attn_desc& d) {
  return size_t(d.batch) * size_t(d.heads_q) * size_t(d.seqlen) * 128;
}

WsLayout ws_layout(const cp_attn_desc& d, const Plan& p, bool backward) {
  WsLayout w;
  size_t off = 256;  // header
  w.tables = off;
  if (!backward) {
    off = align_up(off + p.fwd_table_bytes, 256);
    const size_t rows = size_t(d.batch) * size_t(p.part_rows) * size_t(d.heads_q);
    w.part_o = off;
    off = align_up(off + rows * size_t(d.head_dim) * 4, 256);
    w.part_l = off;
    off = align_up(off + rows * 4, 256);
  } else {
    off = align_up(off + p.bwd_table_bytes, 256);
    const size_t rows = size_t(d.batch) * size_t(d.seqlen) * size_t(d.heads_q);
    w.delta = off;
    off = align_up(off + rows * 4, 256);
    w.lse2 = off;
    off = align_up(off + rows * 4, 256);
    if (d.dtype == CP_BF16 && d.head_dim == 128) {  // tensor-core path: 32-row blocks per (batch, q-head)
      w.dq_acc = off;
      off = align_up(off + dq_acc_floats(d) * 4, 256);
    }
  }
  w.total = off;
  return w;
}

}  // namespace cpattn
