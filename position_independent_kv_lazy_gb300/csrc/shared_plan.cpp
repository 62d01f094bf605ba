// Host planner of the shared-segment decode (lazy_decode_shared_plan).
//
// The position-agnostic pool stores a document once, and every request that retrieves it lists
// the same blocks, each at its own logical offset (LazyAttention summaries, core concept: the
// cache is keyed by content only). In decode the offset only changes the query's rotation
// R(m - o) (decoding part), so two requests holding the same document can attend its pages in
// one pass. The planner finds those shared runs in the host copy of the page tables:
//   - a segment is a maximal run of a request's pages whose offset field repeats (RoPE words
//     carry the segment's offset: one document, or the private tail) or, for ALiBi words (each
//     page's first position, which runs on across documents), advances by the previous page's
//     valid count while the block id advances by one (a document is encoded into consecutive
//     blocks; two documents rarely sit in a context in block order); it is identified by its
//     sequence of (block, valid count) words. Any cut is correct, since the decode takes every
//     row's offset from its own request's word; the cut only decides what can be shared;
//   - identical segments are grouped in order of first appearance, and a group's members are
//     paired in order: (m0, m1), (m2, m3), ...; a leftover member is a single unit, placed right
//     after its group's pairs, so that it re-reads their pages while they are in L2;
//   - units of one group are consecutive, so the decode's warps that run them side by side read
//     the same pages;
//   - a request's segments that no other segment matches (its private tail, documents only it
//     holds) become one single unit per request, after all groups: fewer unit switches, whose
//     query loads stall a warp, and fewer partial slots.
#include <unordered_map>
#include <vector>

#include "pool_internal.h"

namespace {

constexpr uint64_t kOffsetMask = 0x3FFFFFFull << 32;  // page-word bits 32-57

uint32_t offset_of(uint64_t w) { return (uint32_t)((w >> 32) & 0x3FFFFFFu); }
uint32_t nvalid_of(uint64_t w) { return (uint32_t)(w >> 58) + 1u; }

// Page `cur` continues the segment of page `prev`.
bool continues(uint64_t prev, uint64_t cur, bool page_positions) {
  const uint32_t o = offset_of(cur), po = offset_of(prev);
  if (!page_positions) return o == po;
  return o == po + nvalid_of(prev) && (uint32_t)cur == (uint32_t)prev + 1u;
}

struct Segment {
  int32_t req, start, len;
};

// Bucket key of a segment: its length and first (block, valid count) word, through the
// splitmix64 finaliser. A document's first block names it in practice; members of a bucket are
// confirmed word by word, so a collision only costs a comparison.
uint64_t fmix(uint64_t x) {
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ull;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}
uint64_t segment_hash(const uint64_t *words, const Segment &sg) {
  return fmix((words[sg.start] & ~kOffsetMask) ^ ((uint64_t)sg.len * 0x9e3779b97f4a7c15ull));
}
bool same_content(const uint64_t *words, const Segment &a, const Segment &b) {
  if (a.len != b.len) return false;
  for (int32_t k = 0; k < a.len; ++k)
    if ((words[a.start + k] & ~kOffsetMask) != (words[b.start + k] & ~kOffsetMask)) return false;
  return true;
}

}  // namespace

extern "C" int lazy_decode_shared_plan(const uint64_t *words, const int32_t *cu_pages,
                                       int32_t batch, int32_t page_positions,
                                       uint64_t *entries, int32_t *cu_entries,
                                       int32_t *unit_req, int32_t *cu_members, int32_t *members,
                                       int32_t *member_entries, int32_t *n_units,
                                       int32_t *n_entries) {
  if (batch < 0 || !cu_pages || !cu_entries || !cu_members || !n_units || !n_entries)
    return LAZY_ERR_INVALID_ARG;
  for (int32_t b = 0; b < batch; ++b)
    if (cu_pages[b] < 0 || cu_pages[b + 1] < cu_pages[b]) return LAZY_ERR_INVALID_ARG;
  const int32_t total = batch > 0 ? cu_pages[batch] - cu_pages[0] : 0;
  if (total > 0 && (!words || !entries || !unit_req || !members || !member_entries))
    return LAZY_ERR_INVALID_ARG;

  // segments, grouped by content (groups in order of first appearance)
  std::unordered_map<uint64_t, std::vector<int32_t>> index;  // hash -> groups with that hash
  std::vector<std::vector<Segment>> groups;
  for (int32_t b = 0; b < batch; ++b) {
    int32_t k = cu_pages[b];
    const int32_t end = cu_pages[b + 1];
    while (k < end) {
      int32_t e = k + 1;
      while (e < end && continues(words[e - 1], words[e], page_positions != 0)) ++e;
      const Segment sg{b, k, e - k};
      std::vector<int32_t> &bucket = index[segment_hash(words, sg)];
      int32_t gi = -1;
      for (int32_t g : bucket)
        if (same_content(words, groups[g][0], sg)) {
          gi = g;
          break;
        }
      if (gi < 0) {
        gi = (int32_t)groups.size();
        bucket.push_back(gi);
        groups.emplace_back();
      }
      groups[gi].push_back(sg);
      k = e;
    }
  }

  // units: pairs of members of one group, then a leftover single
  std::vector<std::vector<int32_t>> per_req(batch > 0 ? batch : 0);
  int32_t nu = 0, ne = 0;
  cu_entries[0] = 0;
  // unshared segments, per request, for the merged single units at the end
  std::vector<std::vector<Segment>> lone(batch > 0 ? batch : 0);
  for (const auto &grp : groups) {
    if (grp.size() == 1) {
      lone[grp[0].req].push_back(grp[0]);
      continue;
    }
    for (size_t i = 0; i < grp.size(); i += 2) {
      const Segment &a = grp[i];
      const bool pair = i + 1 < grp.size();
      const Segment &bseg = pair ? grp[i + 1] : grp[i];
      for (int32_t k = 0; k < a.len; ++k) {
        entries[2 * (size_t)ne] = words[a.start + k];
        entries[2 * (size_t)ne + 1] = pair ? words[bseg.start + k] : 0ull;
        ++ne;
      }
      unit_req[2 * nu] = a.req;
      unit_req[2 * nu + 1] = pair ? bseg.req : -1;
      per_req[a.req].push_back(2 * nu);
      if (pair) per_req[bseg.req].push_back(2 * nu + 1);
      ++nu;
      cu_entries[nu] = ne;
    }
  }
  for (int32_t b = 0; b < batch; ++b) {
    if (lone[b].empty()) continue;
    for (const Segment &sg : lone[b])
      for (int32_t k = 0; k < sg.len; ++k) {
        entries[2 * (size_t)ne] = words[sg.start + k];
        entries[2 * (size_t)ne + 1] = 0ull;
        ++ne;
      }
    unit_req[2 * nu] = b;
    unit_req[2 * nu + 1] = -1;
    per_req[b].push_back(2 * nu);
    ++nu;
    cu_entries[nu] = ne;
  }
  int32_t nm = 0;
  cu_members[0] = 0;
  for (int32_t b = 0; b < batch; ++b) {
    for (int32_t m : per_req[b]) {
      const int32_t u = m >> 1;
      member_entries[2 * nm] = cu_entries[u];
      member_entries[2 * nm + 1] = cu_entries[u + 1] - cu_entries[u];
      members[nm++] = m;
    }
    cu_members[b + 1] = nm;
  }
  *n_units = nu;
  *n_entries = ne;
  return LAZY_OK;
}
