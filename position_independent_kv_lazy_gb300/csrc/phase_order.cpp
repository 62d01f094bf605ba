// Host scheduling helper: the order of each request's segments for the split-KV decode
// (lazy_order_segments).
//
// The pool caches a retrieved document once and every request that holds it lists the same
// blocks (LazyAttention summaries, core concept: the cache is keyed by content only). Attention
// over a request does not depend on the order of its pages, so the caller may choose it. The
// decode cuts the flattened (request, virtual head, page) sequence into equal contiguous ranges,
// one per warp, and all warps stream their ranges at about the same rate: flattened page x is
// read at about local step x mod R of its range, R = N / ranges. A document shared by several
// requests is read from DRAM once only if those requests reach its pages within a few steps of
// one another, while the pages are still in L2; otherwise each read goes to DRAM again.
//
// For requests whose movable segments all have one page count L, slot k of request b (its k-th
// movable segment) starts at local step phase(b, k, h) = (S_b + h n_b + L k) mod R for virtual
// head h, with S_b the request's first flattened page and n_b its page count. Shared segments are
// placed greedily, most used first: the target is the achievable phase that minimises the summed
// circular distance of all users' best free slots, and each user then takes its best free slot.
// Unshared movable segments fill the remaining slots in their given order; pinned segments (a
// request's private tail) follow, in their given order. Requests with movable segments of
// different page counts keep their given order.
#include <algorithm>
#include <cmath>
#include <unordered_map>
#include <vector>

#include "pool_internal.h"

namespace {

struct Use {
  int32_t req;  // request
  int32_t seg;  // segment index within the request
};

}  // namespace

extern "C" int lazy_order_segments(int32_t batch, const int32_t *cu_segs, const int64_t *seg_key,
                                   const int32_t *seg_pages, const uint8_t *pinned,
                                   int32_t virtual_heads, int64_t ranges, int32_t *perm) {
  if (batch < 0 || !cu_segs || virtual_heads < 1 || ranges < 1) return LAZY_ERR_INVALID_ARG;
  if (cu_segs[0] != 0) return LAZY_ERR_INVALID_ARG;
  for (int32_t b = 0; b < batch; ++b)
    if (cu_segs[b + 1] < cu_segs[b]) return LAZY_ERR_INVALID_ARG;
  const int32_t n_segs = cu_segs[batch];
  if (n_segs > 0 && (!seg_key || !seg_pages || !pinned || !perm)) return LAZY_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_segs; ++i)
    if (seg_pages[i] < 0) return LAZY_ERR_INVALID_ARG;

  // request page counts, flattened starts, the range length
  std::vector<int64_t> n(batch), start(batch);
  int64_t total = 0;
  for (int32_t b = 0; b < batch; ++b) {
    int64_t s = 0;
    for (int32_t i = cu_segs[b]; i < cu_segs[b + 1]; ++i) s += seg_pages[i];
    n[b] = s;
    start[b] = (int64_t)virtual_heads * total;
    total += s;
  }
  const double R = (double)virtual_heads * (double)total / (double)ranges;

  // movable segments per request and their common page count (-1: not uniform)
  std::vector<std::vector<int32_t>> movable(batch);
  std::vector<int64_t> slot_len(batch, 0);
  for (int32_t b = 0; b < batch; ++b) {
    int64_t L = -2;
    for (int32_t i = cu_segs[b]; i < cu_segs[b + 1]; ++i) {
      if (pinned[i]) continue;
      movable[b].push_back(i - cu_segs[b]);
      if (L == -2) L = seg_pages[i];
      else if (L != seg_pages[i]) L = -1;
    }
    slot_len[b] = L;
  }
  // placed[b][k] = segment index at slot k (-1: free)
  std::vector<std::vector<int32_t>> placed(batch);
  for (int32_t b = 0; b < batch; ++b) placed[b].assign(movable[b].size(), -1);

  auto circ = [R](double x) {
    double r = std::fmod(x, R);
    if (r < 0) r += R;
    return std::min(r, R - r);
  };
  // phase distance of (b, k) from (b0, k0), summed over the virtual heads
  auto cost = [&](int32_t b, int64_t k, int32_t b0, int64_t k0) {
    const double base = (double)(start[b] - start[b0]) + (double)(slot_len[b] * k) -
                        (double)(slot_len[b0] * k0);
    const double dh = (double)(n[b] - n[b0]);
    double c = 0.0;
    for (int32_t h = 0; h < virtual_heads; ++h) c += circ(base + dh * h);
    return c;
  };
  auto uniform = [&](int32_t b) { return slot_len[b] >= 0 && R > 0.0; };

  // shared segments: keys used by at least two movable segments of uniform requests
  std::unordered_map<int64_t, std::vector<Use>> users;
  std::vector<int64_t> keys;
  for (int32_t b = 0; b < batch; ++b) {
    if (!uniform(b)) continue;
    for (int32_t s : movable[b]) {
      const int64_t key = seg_key[cu_segs[b] + s];
      auto it = users.find(key);
      if (it == users.end()) {
        keys.push_back(key);
        users[key].push_back({b, s});
      } else {
        it->second.push_back({b, s});
      }
    }
  }
  std::stable_sort(keys.begin(), keys.end(), [&](int64_t a, int64_t c) {
    return users[a].size() > users[c].size();
  });
  std::vector<uint8_t> done(n_segs, 0);
  for (int64_t key : keys) {
    const std::vector<Use> &us = users[key];
    if (us.size() < 2) break;  // sorted by use count: the rest are unshared
    // the target: the (user, free slot) whose phase the users' best free slots sit closest to
    double best = INFINITY;
    int32_t tb = -1;
    int64_t tk = -1;
    for (const Use &u0 : us) {
      for (size_t k0 = 0; k0 < placed[u0.req].size(); ++k0) {
        if (placed[u0.req][k0] >= 0) continue;
        double total_cost = 0.0;
        for (const Use &u : us) {
          double c = INFINITY;
          for (size_t k = 0; k < placed[u.req].size(); ++k)
            if (placed[u.req][k] < 0) c = std::min(c, cost(u.req, (int64_t)k, u0.req, (int64_t)k0));
          if (c < INFINITY) total_cost += c;
        }
        if (total_cost < best) {
          best = total_cost;
          tb = u0.req;
          tk = (int64_t)k0;
        }
      }
    }
    if (tb < 0) continue;
    for (const Use &u : us) {
      int64_t bk = -1;
      double bc = INFINITY;
      for (size_t k = 0; k < placed[u.req].size(); ++k) {
        if (placed[u.req][k] >= 0) continue;
        const double c = cost(u.req, (int64_t)k, tb, tk);
        if (c < bc) {
          bc = c;
          bk = (int64_t)k;
        }
      }
      if (bk >= 0) {
        placed[u.req][bk] = u.seg;
        done[cu_segs[u.req] + u.seg] = 1;
      }
    }
  }
  // output: placed slots (unshared segments fill the free ones in order), then pinned segments
  for (int32_t b = 0; b < batch; ++b) {
    int32_t *out = perm + cu_segs[b];
    int32_t pos = 0;
    if (uniform(b)) {
      size_t next = 0;
      for (size_t k = 0; k < placed[b].size(); ++k) {
        if (placed[b][k] < 0) {
          while (next < movable[b].size() && done[cu_segs[b] + movable[b][next]]) ++next;
          placed[b][k] = movable[b][next];
          done[cu_segs[b] + movable[b][next]] = 1;
        }
        out[pos++] = placed[b][k];
      }
    } else {
      for (int32_t s : movable[b]) out[pos++] = s;
    }
    for (int32_t i = cu_segs[b]; i < cu_segs[b + 1]; ++i)
      if (pinned[i]) out[pos++] = i - cu_segs[b];
  }
  return LAZY_OK;
}
