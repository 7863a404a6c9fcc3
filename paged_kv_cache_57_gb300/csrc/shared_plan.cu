// shared_plan.cu -- host planner of the shared-run decode (decode_shared.cu).
//
// Input: the per-sequence document lists the block-word packer takes. Two
// occurrences (segments) of the same document with the same used length read
// identical physical blocks, whatever their offsets ("Metodologia: Codificação
// Posicional Diferida": the stored keys carry no global position, which is what
// makes them shareable), so they form one group. A group is split into sets of
// at most LAZY_PLAN_MAX_MEMBERS members and at most rows_cap query rows (members x
// query heads per KV head): 64 (RT = 1, 2 or 4 tiles of 16 rows for the mma.sync
// kernel) or 128 (one tensor-core tile). A set's blocks
// are cut into chunks of chunk_blocks logical blocks; each (set, chunk) is one
// item, and every member of the set owns one partial-result slot per chunk. The
// slots of sequence s are slot_indptr[s] .. slot_indptr[s+1]-1. An item also
// carries the physical ids of its first 32 blocks, so the kernel can start its
// loads before the block words arrive.
//
// Items are ordered by decreasing block count, and otherwise keep the order of
// the groups, so items of 1, 2 and 4 row tiles stay mixed through the launch (an
// SM then runs load-bound and tensor-bound items side by side). The items of one
// group stay adjacent, so the CTAs that read the same blocks run at about the
// same time. For the bf16 mma.sync kernel (spread_small), items of at most 8
// blocks are the exception: they are spread evenly through the order (measured:
// 66.0 -> 65.0 us per step on the 8B decode, whose 64-token private tails make 31%
// of the items; the e4m3 instantiation ran slower that way, 75 -> 81 us).
#include <algorithm>
#include <utility>
#include <vector>

#include "kernels.h"

namespace lazy {

int plan_shared_host(int B, int G, int rows_cap, int max_blocks, int num_pool_blocks, int num_docs, const int32_t* seg_indptr,
                     const int32_t* seg_doc, const int32_t* seg_len, const int32_t* doc_block_indptr,
                     const int32_t* doc_blocks, int chunk_blocks, int auto_items, int capacity, int32_t* items,
                     int32_t* slot_indptr, int32_t* counts, bool spread_small) {
  struct Occ {
    int seq, b0;
  };
  const int kBlk = 16;
  // ---- group the occurrences by (document, used length): the groups of document d
  // form a list from doc_head[d] (a document is rarely used at two lengths); each
  // occurrence is tagged with its group, then the groups are laid out contiguously.
  std::vector<int> doc_head(std::max(0, num_docs), -1), group_next;
  std::vector<std::pair<int, int>> keys;  // (doc, len)
  std::vector<int> occ_group;
  std::vector<Occ> occ_all;
  for (int s = 0; s < B; ++s) {
    const int k0 = seg_indptr[s], k1 = seg_indptr[s + 1];
    if (k1 < k0) return LAZY_ERR_LAYOUT;
    int64_t blk = 0;
    for (int k = k0; k < k1; ++k) {
      const int doc = seg_doc[k], len = seg_len[k];
      if (doc < 0 || doc >= num_docs || len < 1) return LAZY_ERR_LAYOUT;
      const int dblk = doc_block_indptr[doc + 1] - doc_block_indptr[doc];
      if ((int64_t)len > (int64_t)kBlk * dblk) return LAZY_ERR_LAYOUT;
      const int nbk = (len + kBlk - 1) / kBlk;
      if (blk + nbk > max_blocks) return LAZY_ERR_LAYOUT;
      for (int q = 0; q < nbk; ++q) {
        const int phys = doc_blocks[doc_block_indptr[doc] + q];
        if (phys < 0 || phys >= num_pool_blocks) return LAZY_ERR_LAYOUT;
      }
      int gi = doc_head[doc];
      while (gi >= 0 && keys[gi].second != len) gi = group_next[gi];
      if (gi < 0) {
        gi = (int)keys.size();
        keys.emplace_back(doc, len);
        group_next.push_back(doc_head[doc]);
        doc_head[doc] = gi;
      }
      occ_group.push_back(gi);
      occ_all.push_back(Occ{s, (int)blk});
      blk += nbk;
    }
  }
  // Occurrences of group gi: occ[gstart[gi] .. gstart[gi + 1]), in input order.
  const int ng = (int)keys.size();
  std::vector<int> gstart(ng + 1, 0);
  for (int g : occ_group) ++gstart[g + 1];
  for (int g = 0; g < ng; ++g) gstart[g + 1] += gstart[g];
  std::vector<Occ> occ(occ_all.size());
  {
    std::vector<int> fill(gstart.begin(), gstart.end() - 1);
    for (size_t k = 0; k < occ_all.size(); ++k) occ[fill[occ_group[k]]++] = occ_all[k];
  }
  auto gsize = [&](int gi) { return gstart[gi + 1] - gstart[gi]; };
  // ---- member sets, their chunk length, and the slots each member needs
  const int per_set = std::max(1, std::min(LAZY_PLAN_MAX_MEMBERS, rows_cap / G));
  struct Set {
    int group, first, n, rt, cb;
  };
  int cb = chunk_blocks;
  if (cb <= 0) {  // about auto_items items: 32 .. 256 blocks, a multiple of 4 (one key tile)
    int64_t total = 0;
    for (int gi = 0; gi < ng; ++gi)
      total += (int64_t)((keys[gi].second + kBlk - 1) / kBlk) * ((gsize(gi) + per_set - 1) / per_set);
    const int64_t per = (total + std::max(1, auto_items) - 1) / std::max(1, auto_items);
    cb = (int)std::min<int64_t>(256, std::max<int64_t>(32, (per + 3) / 4 * 4));
  }
  std::vector<Set> sets;
  std::vector<int> nslots(B, 0);
  for (int gi = 0; gi < ng; ++gi) {
    const int nbk = (keys[gi].second + kBlk - 1) / kBlk;
    for (int j0 = 0; j0 < gsize(gi); j0 += per_set) {
      const int n = std::min(per_set, gsize(gi) - j0);
      const int rows = n * G;
      const int rt = rows <= 16 ? 1 : (rows <= 32 ? 2 : 4);
      sets.push_back(Set{gi, gstart[gi] + j0, n, rt, cb});
      for (int j = 0; j < n; ++j) nslots[occ[gstart[gi] + j0 + j].seq] += (nbk + cb - 1) / cb;
    }
  }
  slot_indptr[0] = 0;
  for (int s = 0; s < B; ++s) slot_indptr[s + 1] = slot_indptr[s] + nslots[s];
  // ---- items, one per (set, chunk)
  struct Item {
    int set, c0, nb, last, cost;
  };
  std::vector<Item> its;
  for (int si = 0; si < (int)sets.size(); ++si) {
    const Set& st = sets[si];
    const int len = keys[st.group].second;
    const int nbk = (len + kBlk - 1) / kBlk;
    for (int c0 = 0; c0 < nbk; c0 += st.cb) {
      const int nb = std::min(st.cb, nbk - c0);
      const int last = (c0 + nb == nbk) ? ((len - 1) & (kBlk - 1)) + 1 : kBlk;
      its.push_back(Item{si, c0, nb, last, nb});
    }
  }
  if ((int64_t)its.size() > capacity) return LAZY_ERR_WORKSPACE;
  std::stable_sort(its.begin(), its.end(), [](const Item& x, const Item& y) { return x.cost > y.cost; });
  // Items of at most kSmall blocks (a sequence's private tail, say) cost an item's fixed
  // latency for little data; spread evenly through the launch instead of ending it, they
  // run beside streaming items, and the launch does not end on a wave of them.
  if (spread_small) {
    constexpr int kSmall = 8;
    std::vector<Item> big, small;
    for (const Item& it : its) (it.nb <= kSmall ? small : big).push_back(it);
    if (!small.empty() && !big.empty()) {
      const size_t n = its.size();
      size_t bi = 0, si = 0;
      for (size_t k = 0; k < n; ++k) {
        // small item si goes to position floor((si + 0.5) * n / small.size())
        const bool take_small =
            si < small.size() && (bi >= big.size() || (double)k >= ((double)si + 0.5) * (double)n / (double)small.size());
        its[k] = take_small ? small[si++] : big[bi++];
      }
    }
  }
  std::vector<int> next(slot_indptr, slot_indptr + B);
  for (size_t i = 0; i < its.size(); ++i) {
    const Set& st = sets[its[i].set];
    int32_t* d = items + (size_t)LAZY_PLAN_ITEM_INTS * i;
    std::fill(d, d + LAZY_PLAN_ITEM_INTS, 0);
    d[0] = occ[st.first].seq;
    d[1] = occ[st.first].b0 + its[i].c0;
    d[2] = its[i].nb;
    d[3] = its[i].last;
    d[4] = st.n;
    d[5] = its[i].c0;  // the item's first block within its document
    for (int j = 0; j < st.n; ++j) {
      const Occ& o = occ[st.first + j];
      int32_t* m = d + 8 + 4 * j;
      m[0] = o.seq;
      m[1] = o.b0 + its[i].c0;
      m[2] = next[o.seq]++;
    }
    const int doc = keys[st.group].first;
    int32_t* ids = d + 8 + 4 * LAZY_PLAN_MAX_MEMBERS;
    for (int k = 0; k < its[i].nb && k < LAZY_PLAN_ITEM_BLOCK_IDS; ++k)
      ids[k] = doc_blocks[doc_block_indptr[doc] + its[i].c0 + k];
  }
  counts[0] = (int32_t)its.size();
  counts[1] = slot_indptr[B];
  return LAZY_OK;
}

}  // namespace lazy
