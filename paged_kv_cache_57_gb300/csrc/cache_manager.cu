// cache_manager.cu -- host-side cache manager for the paged KV pool and the policy
// replay simulator declared in include/lazy_cache.h (no device code).
//
// Blocks come from a free list ("KV Cache, Flash Attention & Otimização de
// Inferência", "PagedAttention": 16-token blocks, a free list, blocks returned to
// the pool when no longer needed). Cached runs are entries keyed by the policy:
// the document alone (position-agnostic, the LazyAttention cache of "Resumo
// Técnico: LazyAttention", "Metodologia"), the document and its offset
// (position-aware: one stored variant per position, "Declaração do Problema"), or
// the whole preceding request prefix (prefix caching). Entries pinned by admitted
// requests are never evicted; the others leave least-recently-used first.
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/lazy_attn.h"
#include "../../include/lazy_cache.h"

namespace {

constexpr int kBlk = 16;

struct Entry {
  uint64_t key = 0;
  // identity checked on every hit (the key is only its hash for prefix caching)
  int32_t doc = 0, offset = 0;
  uint64_t parent = 0;
  int32_t tokens = 0;
  std::vector<int32_t> blocks;
  int32_t pins = 0;
  bool in_map = true;                        // false: replaced, freed at its last release
  std::list<Entry*>::iterator lru;           // valid while in_map
};

uint64_t mix64(uint64_t x) {  // splitmix64 finaliser
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

int32_t blocks_of(int32_t len) { return (len + kBlk - 1) / kBlk; }

}  // namespace

struct lazy_cache {
  int32_t policy = 0;
  // Free ids: a stack of returned ids (the most recently freed is reused first) above
  // the never-used ids next_fresh .. num_blocks-1, handed out in increasing order.
  std::vector<int32_t> free_list;
  int32_t num_blocks = 0, next_fresh = 0;
  std::unordered_map<uint64_t, Entry*> map;
  std::list<Entry*> lru;  // front: least recently used
  std::unordered_map<int64_t, std::vector<Entry*>> tickets;
  int64_t next_ticket = 1;
  lazy_cache_stats st{};

  ~lazy_cache() {
    std::unordered_set<Entry*> orphans;  // replaced entries still pinned: reachable only from tickets
    for (auto& kv : tickets)
      for (Entry* e : kv.second)
        if (!e->in_map) orphans.insert(e);
    for (auto& kv : map) delete kv.second;
    for (Entry* e : orphans) delete e;
  }

  // Key and identity of segment (doc, len) at `offset`, after the prefix hash `chain`.
  uint64_t key_of(int32_t doc, int32_t len, int32_t offset, uint64_t chain) const {
    if (policy == LAZY_CACHE_POSITION_AGNOSTIC) return (uint64_t)(uint32_t)doc;
    if (policy == LAZY_CACHE_POSITION_AWARE) return ((uint64_t)(uint32_t)doc << 32) | (uint32_t)offset;
    return mix64(chain ^ mix64(((uint64_t)(uint32_t)doc << 32) | (uint32_t)len));
  }
  bool same(const Entry* e, int32_t doc, int32_t len, int32_t offset, uint64_t chain) const {
    if (e->doc != doc) return false;
    if (policy == LAZY_CACHE_POSITION_AGNOSTIC) return e->tokens >= len;
    if (policy == LAZY_CACHE_POSITION_AWARE) return e->offset == offset && e->tokens >= len;
    return e->parent == chain && e->tokens == len;
  }

  int64_t free_count() const { return (int64_t)free_list.size() + (num_blocks - next_fresh); }
  int32_t take_block() {
    if (free_list.empty()) return next_fresh++;
    const int32_t b = free_list.back();
    free_list.pop_back();
    return b;
  }
  void free_entry_blocks(Entry* e) {
    for (int32_t b : e->blocks) free_list.push_back(b);
    st.resident_blocks -= (int64_t)e->blocks.size();
    e->blocks.clear();
  }
  void evict(Entry* e) {  // unpinned entry in the map
    st.evicted_blocks += (int64_t)e->blocks.size();
    free_entry_blocks(e);
    lru.erase(e->lru);
    map.erase(e->key);
    delete e;
  }
  void unpin(Entry* e) {
    if (--e->pins == 0 && !e->in_map) {
      st.evicted_blocks += (int64_t)e->blocks.size();
      free_entry_blocks(e);
      delete e;
    }
  }
  void touch(Entry* e) { lru.splice(lru.end(), lru, e->lru); }
};

extern "C" {

lazy_cache* lazy_cache_create(int32_t num_blocks, int32_t policy) {
  if (num_blocks <= 0 || policy < LAZY_CACHE_POSITION_AGNOSTIC || policy > LAZY_CACHE_PREFIX) return nullptr;
  lazy_cache* c = new (std::nothrow) lazy_cache;
  if (!c) return nullptr;
  c->policy = policy;
  c->num_blocks = num_blocks;  // id 0 is handed out first
  return c;
}

void lazy_cache_destroy(lazy_cache* c) { delete c; }

int lazy_cache_admit(lazy_cache* c, int32_t nseg, const int32_t* seg_doc, const int32_t* seg_len, int32_t pos0,
                     int32_t* out_indptr, int32_t* out_blocks, int32_t capacity, int32_t* out_hit,
                     int64_t* ticket) {
  if (!c || nseg < 0 || pos0 < 0 || !out_indptr || !ticket || capacity < 0) return LAZY_ERR_INVALID_ARG;
  if (nseg > 0 && (!seg_doc || !seg_len || !out_hit)) return LAZY_ERR_INVALID_ARG;
  int64_t need_out = 0, end = pos0;
  for (int32_t i = 0; i < nseg; ++i) {
    if (seg_doc[i] < 0 || seg_len[i] < 1) return LAZY_ERR_INVALID_ARG;
    need_out += blocks_of(seg_len[i]);
    end += seg_len[i];
  }
  if (end > INT32_MAX) return LAZY_ERR_INVALID_ARG;
  if (need_out > capacity || (need_out > 0 && !out_blocks)) return LAZY_ERR_WORKSPACE;

  // Phase 1: hits (pinned at once, so no eviction below can take them) and misses.
  // A segment repeated within the request hits the entry its first occurrence creates.
  struct Plan {
    uint64_t key, chain;
    int32_t offset;
    Entry* hit;
    int32_t first_miss;  // index of the earlier miss it reuses, or -1
  };
  std::vector<Plan> plan((size_t)nseg);
  std::unordered_map<uint64_t, int32_t> new_keys;  // key -> first segment that creates it
  int64_t new_blocks = 0;
  uint64_t chain = mix64((uint64_t)(uint32_t)pos0);
  int32_t offset = pos0;
  std::vector<Entry*> pinned;
  for (int32_t i = 0; i < nseg; ++i) {
    Plan& pl = plan[(size_t)i];
    pl.chain = chain;
    pl.offset = offset;
    pl.key = c->key_of(seg_doc[i], seg_len[i], offset, chain);
    pl.hit = nullptr;
    pl.first_miss = -1;
    auto nk = new_keys.find(pl.key);
    if (nk != new_keys.end() && c->policy != LAZY_CACHE_PREFIX && seg_len[i] <= seg_len[nk->second] &&
        seg_doc[i] == seg_doc[nk->second]) {
      pl.first_miss = nk->second;
    } else {
      auto f = c->map.find(pl.key);
      if (f != c->map.end() && c->same(f->second, seg_doc[i], seg_len[i], offset, chain)) {
        pl.hit = f->second;
        ++pl.hit->pins;
        pinned.push_back(pl.hit);
      } else {
        new_keys[pl.key] = i;
        new_blocks += blocks_of(seg_len[i]);
      }
    }
    if (c->policy == LAZY_CACHE_PREFIX) chain = pl.key;
    offset += seg_len[i];
  }
  // Phase 2: room for the new blocks. A request that would not fit even with every
  // unpinned entry evicted is refused before anything is evicted; otherwise unpinned
  // entries leave least-recently-used first (entries about to be replaced go the
  // same way).
  if (c->free_count() < new_blocks) {
    int64_t avail = c->free_count();
    for (const Entry* e : c->lru)
      if (e->pins == 0) avail += (int64_t)e->blocks.size();
    if (avail < new_blocks) {
      for (Entry* e : pinned) c->unpin(e);
      ++c->st.rejected;
      return LAZY_ERR_LAYOUT;
    }
  }
  for (auto it = c->lru.begin(); c->free_count() < new_blocks;) {
    Entry* e = *it;
    ++it;
    if (e->pins == 0) c->evict(e);
  }
  // Phase 3: new entries (replacing any stale entry under the same key).
  std::vector<Entry*> made((size_t)nseg, nullptr);
  for (int32_t i = 0; i < nseg; ++i) {
    Plan& pl = plan[(size_t)i];
    if (pl.hit || pl.first_miss >= 0) continue;
    auto f = c->map.find(pl.key);
    if (f != c->map.end()) {
      Entry* old = f->second;
      if (old->pins == 0) {
        c->evict(old);
      } else {  // still in use: leaves the map, freed at its last release
        old->in_map = false;
        c->lru.erase(old->lru);
        c->map.erase(f);
      }
    }
    Entry* e = new Entry;
    e->key = pl.key;
    e->doc = seg_doc[i];
    e->offset = pl.offset;
    e->parent = pl.chain;
    e->tokens = seg_len[i];
    const int32_t nb = blocks_of(seg_len[i]);
    e->blocks.resize((size_t)nb);
    for (int32_t k = 0; k < nb; ++k) e->blocks[(size_t)k] = c->take_block();
    c->st.resident_blocks += nb;
    if (c->st.resident_blocks > c->st.peak_resident_blocks) c->st.peak_resident_blocks = c->st.resident_blocks;
    e->lru = c->lru.insert(c->lru.end(), e);
    c->map[pl.key] = e;
    e->pins = 1;
    pinned.push_back(e);
    made[(size_t)i] = e;
  }
  // Outputs, pins of repeated segments, recency.
  int32_t pos = 0;
  for (int32_t i = 0; i < nseg; ++i) {
    Plan& pl = plan[(size_t)i];
    Entry* e = pl.hit ? pl.hit : (pl.first_miss >= 0 ? made[(size_t)pl.first_miss] : made[(size_t)i]);
    if (pl.first_miss >= 0) {
      ++e->pins;
      pinned.push_back(e);
    }
    const int32_t nb = blocks_of(seg_len[i]);
    out_indptr[i] = pos;
    for (int32_t k = 0; k < nb; ++k) out_blocks[pos + k] = e->blocks[(size_t)k];
    pos += nb;
    const bool hit = pl.hit != nullptr || pl.first_miss >= 0;
    out_hit[i] = hit ? 1 : 0;
    (hit ? c->st.hit_blocks : c->st.miss_blocks) += nb;
    if (e->in_map) c->touch(e);
  }
  out_indptr[nseg] = pos;
  *ticket = c->next_ticket++;
  c->tickets.emplace(*ticket, std::move(pinned));
  return LAZY_OK;
}

int lazy_cache_release(lazy_cache* c, int64_t ticket) {
  if (!c) return LAZY_ERR_INVALID_ARG;
  auto f = c->tickets.find(ticket);
  if (f == c->tickets.end()) return LAZY_ERR_INVALID_ARG;
  std::vector<Entry*> pins = std::move(f->second);
  c->tickets.erase(f);
  for (Entry* e : pins) c->unpin(e);
  return LAZY_OK;
}

int lazy_cache_get_stats(const lazy_cache* c, lazy_cache_stats* out) {
  if (!c || !out) return LAZY_ERR_INVALID_ARG;
  *out = c->st;
  return LAZY_OK;
}

int lazy_cache_simulate(int32_t policy, int32_t num_blocks, int32_t num_requests, const int32_t* seg_indptr,
                        const int32_t* seg_doc, const int32_t* seg_len, const int32_t* pos0, int32_t concurrency,
                        lazy_cache_stats* out) {
  if (num_requests < 0 || concurrency < 1 || !out || (num_requests > 0 && !seg_indptr)) return LAZY_ERR_INVALID_ARG;
  for (int32_t r = 0; r < num_requests; ++r)
    if (seg_indptr[r + 1] < seg_indptr[r]) return LAZY_ERR_INVALID_ARG;
  lazy_cache* c = lazy_cache_create(num_blocks, policy);
  if (!c) return LAZY_ERR_INVALID_ARG;
  std::vector<int64_t> live;  // tickets in admission order (0: rejected)
  std::vector<int32_t> indptr, blocks, hit;
  int rc = LAZY_OK;
  for (int32_t r = 0; r < num_requests && rc == LAZY_OK; ++r) {
    const int32_t k0 = seg_indptr[r], n = seg_indptr[r + 1] - k0;
    int64_t cap = 0;
    for (int32_t k = k0; k < k0 + n; ++k) cap += seg_len[k] > 0 ? blocks_of(seg_len[k]) : 0;
    indptr.assign((size_t)n + 1, 0);
    blocks.assign((size_t)(cap > 0 ? cap : 1), 0);
    hit.assign((size_t)(n > 0 ? n : 1), 0);
    int64_t t = 0;
    const int a = lazy_cache_admit(c, n, seg_doc + k0, seg_len + k0, pos0 ? pos0[r] : 0, indptr.data(), blocks.data(),
                                   (int32_t)cap, hit.data(), &t);
    if (a == LAZY_OK) {
      live.push_back(t);
    } else if (a == LAZY_ERR_LAYOUT) {
      live.push_back(0);
    } else {
      rc = a;
    }
    if (live.size() >= (size_t)concurrency) {  // keep at most `concurrency` requests pinned
      int64_t& old = live[live.size() - (size_t)concurrency];
      if (old) lazy_cache_release(c, old);
      old = 0;
    }
  }
  for (int64_t t : live)
    if (t) lazy_cache_release(c, t);
  lazy_cache_get_stats(c, out);
  lazy_cache_destroy(c);
  return rc;
}

}  // extern "C"
