/* lazy_cache.h -- host-side cache manager for a paged KV pool of 16-token blocks,
 * and a replay simulator that compares cache-reuse policies on a request trace.
 *
 * What it models ("Resumo Técnico: LazyAttention", "Declaração do Problema" and
 * "Eficiência de Cache"; "KV Cache, Flash Attention & Otimização de Inferência",
 * "PagedAttention" and its free-list exercise):
 *  - a pool of num_blocks physical blocks handed out from a free list and
 *    returned to it on eviction;
 *  - cached document runs ("entries"): a request is a list of segments
 *    (doc, len) -- the first len tokens of document doc -- placed at concatenated
 *    offsets from pos0. A segment whose entry is cached (and at least len tokens
 *    long) reuses that entry's first ceil(len/16) blocks (a hit, counted in
 *    blocks); otherwise its blocks are allocated and must be filled (a miss);
 *  - an entry is pinned while a request that uses it is admitted, and entries
 *    that no admitted request pins are evicted least-recently-used first when the
 *    pool runs short.
 * The policy decides which segments may share an entry:
 *  - LAZY_CACHE_POSITION_AGNOSTIC: the entry of a document serves it at any offset
 *    (stored keys carry no position: the LazyAttention cache);
 *  - LAZY_CACHE_POSITION_AWARE: an entry serves only the same document at the same
 *    offset (keys stored with their absolute positions; one copy per offset);
 *  - LAZY_CACHE_PREFIX: an entry serves only the same segment after the same
 *    preceding segments from the same pos0 (prefix caching).
 * Status codes are those of lazy_attn.h. All calls are host-only, single-threaded
 * per cache object, and allocate with the C++ heap (never device memory).
 */
#ifndef LAZY_CACHE_H
#define LAZY_CACHE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LAZY_CACHE_POSITION_AGNOSTIC 0
#define LAZY_CACHE_POSITION_AWARE 1
#define LAZY_CACHE_PREFIX 2

typedef struct lazy_cache lazy_cache; /* opaque */

/* Counters of a cache (cumulative since creation). */
typedef struct {
  int64_t hit_blocks;       /* blocks of admitted segments found cached */
  int64_t miss_blocks;      /* blocks of admitted segments allocated and filled */
  int64_t evicted_blocks;   /* blocks returned to the free list by eviction */
  int64_t rejected;         /* admissions refused: not enough unpinned blocks */
  int64_t resident_blocks;  /* blocks held by entries now */
  int64_t peak_resident_blocks;
} lazy_cache_stats;

/* A cache over num_blocks (> 0) physical block ids 0 .. num_blocks-1 under
 * `policy`. Returns NULL on a bad argument or allocation failure. */
lazy_cache *lazy_cache_create(int32_t num_blocks, int32_t policy);
void lazy_cache_destroy(lazy_cache *c);

/* Admits one request of nseg segments (seg_doc[i] >= 0, seg_len[i] >= 1 tokens)
 * placed at concatenated offsets from pos0 >= 0. On success every segment's
 * physical block ids (ceil(len/16) of them, in order) are written to
 * out_blocks[out_indptr[i] .. out_indptr[i+1]-1] (out_indptr has nseg+1 entries,
 * out_blocks room for `capacity` ids), out_hit[i] is 1 where the segment reused a
 * cached entry and 0 where its blocks were just allocated (their contents must be
 * computed by the caller), and *ticket identifies the request for
 * lazy_cache_release. The segments' entries stay pinned until then.
 * Returns LAZY_OK (0); LAZY_ERR_INVALID_ARG (1) on bad arguments;
 * LAZY_ERR_WORKSPACE (3) when `capacity` is too small; LAZY_ERR_LAYOUT (4) when
 * the pool cannot hold the request's new blocks even after evicting every
 * unpinned entry (nothing is admitted then, and `rejected` counts it). */
int lazy_cache_admit(lazy_cache *c, int32_t nseg, const int32_t *seg_doc, const int32_t *seg_len, int32_t pos0,
                     int32_t *out_indptr, int32_t *out_blocks, int32_t capacity, int32_t *out_hit,
                     int64_t *ticket);

/* Unpins the entries of an admitted request. LAZY_ERR_INVALID_ARG for an unknown
 * or already released ticket. */
int lazy_cache_release(lazy_cache *c, int64_t ticket);

int lazy_cache_get_stats(const lazy_cache *c, lazy_cache_stats *out);

/* Replays a trace through a fresh cache of num_blocks blocks under `policy`:
 * request r is segments seg_indptr[r] .. seg_indptr[r+1]-1 (seg_indptr has
 * num_requests+1 entries) from position pos0[r] (pos0 NULL: 0). Requests are
 * admitted in order; request r is released right after request
 * r + concurrency - 1 has been admitted (concurrency >= 1; the last ones at the
 * end), so that at most `concurrency` requests pin entries at once. A request that
 * cannot be admitted is counted in `rejected` and skipped. Writes the final
 * counters to *out. Returns the first error of an admission other than
 * LAZY_ERR_LAYOUT, which stops the replay (the counters so far are written). */
int lazy_cache_simulate(int32_t policy, int32_t num_blocks, int32_t num_requests, const int32_t *seg_indptr,
                        const int32_t *seg_doc, const int32_t *seg_len, const int32_t *pos0, int32_t concurrency,
                        lazy_cache_stats *out);

#ifdef __cplusplus
}
#endif

#endif /* LAZY_CACHE_H */
