// Hybrid context parallelism: per-sub-sequence CP sizes on aligned
// power-of-two rank groups, scheduled in rounds ("04 · Megatron-LM 实现" §7.1,
// the balanced scheduler; §2.3, groups are contiguous blocks of ranks aligned
// to their power-of-two size; §1.1, a sequence is split by the zigzag rule
// over its group).  Host only.
//
// A round is built from the pending sequences, longest first:
//  - cost of a sequence on g ranks: len^2 / g (the page's proxy);
//  - ranks it needs: the smallest power of two g with len <= g * capacity;
//  - buckets: one per distinct need, each aiming at total cost / buckets and
//    closed once the next sequence would take it past 1.1x that share;
//  - placement: the least loaded existing group of the sequence's size that
//    still has room for len / g tokens per rank, else a new group on the
//    lowest aligned block of idle ranks, else the sequence waits;
//  - early stop at a bucket step when every rank is busy and the rank loads
//    are within 5% (max - min <= max / 20);
//  - trim: the last placed sequence waits while it sits on a most loaded
//    group and dropping it strictly cuts the slack (max - min over the busy
//    ranks' loads);
//  - merge: the most loaded group whose aligned buddy block is idle doubles
//    (its sequences are split over twice the ranks), until none can.
// Ties go to the lower rank.  Costs are exact integers (lengths are multiples
// of 2 * world), compared in 128-bit arithmetic.
#include <algorithm>
#include <vector>

#include "cpattn.h"

namespace {

struct Group {
  int32_t rank0 = 0, size = 0;
  std::vector<int32_t> seqs;  // in placement order
  bool live() const { return !seqs.empty(); }
};

int64_t cost(int64_t len, int64_t g) { return len * len / g; }

struct Round {
  const std::vector<int64_t>& len;
  const std::vector<int32_t>& need;
  int32_t world;
  int64_t capacity;
  std::vector<Group> groups;
  std::vector<int32_t> owner;  // group index per rank, -1 idle

  int64_t load(const Group& g) const {
    int64_t x = 0;
    for (int32_t k : g.seqs) x += cost(len[k], g.size);
    return x;
  }
  int64_t tokens(const Group& g) const {
    int64_t x = 0;
    for (int32_t k : g.seqs) x += len[k] / g.size;
    return x;
  }
  int64_t slack() const {
    int64_t lo = 0, hi = 0;
    bool any = false;
    for (const Group& g : groups) {
      if (!g.live()) continue;
      const int64_t x = load(g);
      lo = any ? std::min(lo, x) : x;
      hi = any ? std::max(hi, x) : x;
      any = true;
    }
    return hi - lo;
  }
  bool idle(int32_t r0, int32_t n) const {
    for (int32_t r = r0; r < r0 + n; ++r)
      if (owner[r] >= 0) return false;
    return true;
  }
  void take(int32_t gi) {
    for (int32_t r = groups[gi].rank0; r < groups[gi].rank0 + groups[gi].size; ++r) owner[r] = gi;
  }
  void release(int32_t gi) {
    for (int32_t r = groups[gi].rank0; r < groups[gi].rank0 + groups[gi].size; ++r) owner[r] = -1;
  }
};

// Builds one round from `pending` (sorted longest first); `left` receives
// the sequences for later rounds, `cp`/`rank0` the placement of the others.
void build_round(const std::vector<int32_t>& pending, Round& R, std::vector<int32_t>& left,
                 std::vector<std::pair<int32_t, int32_t>>& placed_at, std::vector<int32_t>& placed_seq) {
  const auto& len = R.len;
  const auto& need = R.need;
  // buckets
  std::vector<int32_t> distinct;
  __int128 total = 0;
  for (int32_t k : pending) {
    distinct.push_back(need[k]);
    total += cost(len[k], need[k]);
  }
  std::sort(distinct.begin(), distinct.end());
  const int64_t nb = std::unique(distinct.begin(), distinct.end()) - distinct.begin();
  std::vector<int32_t> bucket(pending.size());
  {
    int32_t b = 0;
    __int128 acc = 0;
    for (size_t i = 0; i < pending.size(); ++i) {
      const int64_t w = cost(len[pending[i]], need[pending[i]]);
      if (acc > 0 && b < nb - 1 && __int128(10) * nb * (acc + w) > __int128(11) * total) {
        ++b;
        acc = 0;
      }
      bucket[i] = b;
      acc += w;
    }
  }

  std::vector<int32_t> order;  // placement order
  for (size_t i = 0; i < pending.size(); ++i) {
    const int32_t k = pending[i];
    if (i > 0 && bucket[i] != bucket[i - 1]) {
      bool all_busy = true;
      int64_t lo = 0, hi = 0;
      for (int32_t r = 0; r < R.world; ++r) {
        if (R.owner[r] < 0) {
          all_busy = false;
          break;
        }
        const int64_t x = R.load(R.groups[R.owner[r]]);
        lo = r == 0 ? x : std::min(lo, x);
        hi = r == 0 ? x : std::max(hi, x);
      }
      if (all_busy && 20 * (hi - lo) <= hi) {
        left.insert(left.end(), pending.begin() + i, pending.end());
        break;
      }
    }
    const int32_t g = need[k];
    int32_t best = -1;
    int64_t best_load = 0;
    for (size_t gi = 0; gi < R.groups.size(); ++gi) {
      const Group& G = R.groups[gi];
      if (!G.live() || G.size != g || R.tokens(G) + len[k] / g > R.capacity) continue;
      const int64_t x = R.load(G);
      if (best < 0 || x < best_load || (x == best_load && G.rank0 < R.groups[best].rank0)) {
        best = int32_t(gi);
        best_load = x;
      }
    }
    if (best < 0) {
      for (int32_t r0 = 0; r0 < R.world; r0 += g) {
        if (R.idle(r0, g)) {
          Group G;
          G.rank0 = r0;
          G.size = g;
          R.groups.push_back(G);
          best = int32_t(R.groups.size()) - 1;
          R.take(best);
          break;
        }
      }
    }
    if (best < 0) {
      left.push_back(k);
      continue;
    }
    R.groups[best].seqs.push_back(k);
    order.push_back(k);
  }

  // trim
  while (order.size() > 1) {
    const int32_t k = order.back();
    int32_t gi = -1;
    for (size_t j = 0; j < R.groups.size() && gi < 0; ++j)
      if (!R.groups[j].seqs.empty() && R.groups[j].seqs.back() == k) gi = int32_t(j);
    const int64_t before = R.slack();
    int64_t top = 0;
    for (const Group& G : R.groups)
      if (G.live()) top = std::max(top, R.load(G));
    if (R.load(R.groups[gi]) < top) break;  // only an overloaded group sheds
    R.groups[gi].seqs.pop_back();
    if (R.slack() < before) {
      order.pop_back();
      left.push_back(k);
      if (!R.groups[gi].live()) R.release(gi);
    } else {
      R.groups[gi].seqs.push_back(k);
      break;
    }
  }

  // merge idle ranks into the most loaded growable group
  for (;;) {
    int32_t pick = -1;
    int64_t pick_load = 0;
    for (size_t gi = 0; gi < R.groups.size(); ++gi) {
      const Group& G = R.groups[gi];
      if (!G.live() || 2 * int64_t(G.size) > R.world || !R.idle(G.rank0 ^ G.size, G.size)) continue;
      const int64_t x = R.load(G);
      if (pick < 0 || x > pick_load || (x == pick_load && G.rank0 < R.groups[pick].rank0)) {
        pick = int32_t(gi);
        pick_load = x;
      }
    }
    if (pick < 0) break;
    Group& G = R.groups[pick];
    G.rank0 = std::min(G.rank0, G.rank0 ^ G.size);
    G.size *= 2;
    R.take(pick);
  }

  for (const Group& G : R.groups)
    for (int32_t k : G.seqs) {
      placed_seq.push_back(k);
      placed_at.push_back({G.size, G.rank0});
    }
}

}  // namespace

extern "C" cp_status cp_hybrid_schedule(const int32_t* lens, int32_t n, int32_t world, int64_t capacity,
                                        int32_t* round, int32_t* cp, int32_t* rank0, int32_t* n_rounds) {
  if (n < 0 || world < 1 || (world & (world - 1)) || capacity < 1 || !n_rounds) return CP_ERR_INVALID_ARG;
  if (n > 0 && (!lens || !round || !cp || !rank0)) return CP_ERR_INVALID_ARG;
  std::vector<int64_t> len(n);
  std::vector<int32_t> need(n);
  for (int32_t k = 0; k < n; ++k) {
    if (lens[k] < 0) return CP_ERR_INVALID_ARG;
    if (lens[k] % (2 * int64_t(world))) return CP_ERR_ALIGNMENT;
    len[k] = lens[k];
    int64_t g = 1;
    while (g * capacity < len[k]) g *= 2;
    if (g > world) return CP_ERR_UNSUPPORTED;
    need[k] = int32_t(g);
  }
  auto longest_first = [&](int32_t a, int32_t b) { return len[a] != len[b] ? len[a] > len[b] : a < b; };
  std::vector<int32_t> pending(n);
  for (int32_t k = 0; k < n; ++k) pending[k] = k;
  std::sort(pending.begin(), pending.end(), longest_first);
  int32_t r = 0;
  while (!pending.empty()) {
    Round R{len, need, world, capacity, {}, std::vector<int32_t>(world, -1)};
    std::vector<int32_t> left, seq;
    std::vector<std::pair<int32_t, int32_t>> at;
    build_round(pending, R, left, at, seq);
    if (seq.empty()) return CP_ERR_UNSUPPORTED;  // no progress (cannot happen for valid input)
    for (size_t i = 0; i < seq.size(); ++i) {
      round[seq[i]] = r;
      cp[seq[i]] = at[i].first;
      rank0[seq[i]] = at[i].second;
    }
    std::sort(left.begin(), left.end(), longest_first);
    pending.swap(left);
    ++r;
  }
  *n_rounds = r;
  return CP_OK;
}
