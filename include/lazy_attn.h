/*
 * lazy_attn.h -- C ABI of a LazyAttention library for one NVIDIA GB300 (sm_103a).
 *
 * LazyAttention (technical summary "Resumo Técnico: LazyAttention", gist.science,
 * paper 2606.04302) keeps the KV cache position-agnostic: each cached document's
 * K rows are stored once, rotated at the document's own local positions
 * 0..len-1, V unrotated, in 16-token physical blocks ("KV Cache, Flash Attention
 * & Otimização de Inferência", section "PagedAttention"). Position is applied on
 * the fly inside the attention kernel ("Metodologia: Codificação Posicional
 * Diferida"): RoPE scores depend only on the relative offset,
 * <R_m q, R_p k> = <R_{m-p} q, k> ("Equivalência Matemática").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: every tensor is allocated and owned by the caller. Pointers named
 *    `*_host` are host memory; every other tensor pointer is device memory of
 *    the current CUDA device. The library allocates no device memory. Its only
 *    global state is one status word per device (see lazy_attn_device_status).
 *  - Asynchrony: compute calls only enqueue kernels on `stream` and return; they
 *    are re-entrant.
 *  - Errors: argument and layout errors that can be seen on the host are
 *    returned synchronously, and nothing is launched. A failed launch returns
 *    LAZY_ERR_CUDA. Conditions that are only visible on the device (a block id
 *    outside the pool, a position outside the rotation table, a pipeline wait
 *    that timed out, a layout error found by the device packer) never trap:
 *    the kernel skips the offending access, sets a bit in the device status
 *    word and returns. Outputs are then unspecified.
 *  - Numerics: dtype LAZY_F32 computes in fp32; LAZY_BF16 multiplies bf16
 *    operands on the tensor cores with fp32 accumulation and fp32 softmax.
 *    With kv_dtype LAZY_FP8_E4M3 (the decodes: lazy_attn_decode, _noalloc and
 *    lazy_attn_decode_shared) the pools hold OCP e4m3 codes and the products take
 *    f16 operands (every e4m3 value is exact in f16), with fp32 accumulation and
 *    softmax.
 *
 * Layout (one layer)
 * ------------------
 *  k_pool, v_pool  [num_pool_blocks][num_kv_heads][16][head_dim], dtype. One
 *                  (block, head) is 16*head_dim contiguous elements.
 *  block_words     [num_seqs][max_blocks_per_seq] uint32, one word per logical
 *                  block b of a sequence ("Implementação Técnica", Decoding:
 *                  block ID and offset packed in one register):
 *                      word = ((uint32)off << id_bits) | phys_id
 *                  phys_id = physical block index (low id_bits bits);
 *                  off = 16*b - p as a signed (32-id_bits)-bit two's complement
 *                  field, where p is the global start position of the document
 *                  that block b belongs to. The kernel recovers p = 16*b - off.
 *                  Storing the block-relative form keeps both fields in 32 bits
 *                  for pools of up to 2^id_bits blocks and contexts of 2^17+
 *                  tokens.
 *  seq_lens        [num_seqs] int32. A sequence spans nb = ceil(seq_lens/16)
 *                  logical blocks. Every document starts a fresh logical block,
 *                  so a document whose length is not a multiple of 16 leaves
 *                  unused slots at the end of its last block. Valid slots of
 *                  block b: seq_lens - 16*(nb-1) if b == nb-1; else
 *                  ((p_{b+1} - p_b - 1) & 15) + 1 if p_{b+1} != p_b; else 16.
 *                  Documents of a sequence are contiguous in position
 *                  (p_next = p + used length) and each is used from its first
 *                  token (a prefix is allowed).
 *  RoPE            rotate-half pairs (i, i + head_dim/2), frequencies
 *                  w_i = rope_theta^(-2i/head_dim).
 */
#ifndef LAZY_ATTN_H_
#define LAZY_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *lazy_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  LAZY_OK = 0,
  LAZY_ERR_INVALID_ARG = 1, /* null pointer, bad size or head count */
  LAZY_ERR_UNSUPPORTED = 2, /* a shape or dtype the library has no kernel for */
  LAZY_ERR_WORKSPACE = 3,   /* workspace or table buffer too small */
  LAZY_ERR_LAYOUT = 4,      /* documents/blocks do not form a valid block table */
  LAZY_ERR_CUDA = 5,        /* a CUDA call or launch failed */
  LAZY_ERR_DEVICE = 6       /* the device status word reported a fault */
} lazy_status;

typedef enum { LAZY_F32 = 0, LAZY_BF16 = 1, LAZY_FP8_E4M3 = 2 } lazy_dtype;

/* Bits of the per-device status word. */
#define LAZY_DEV_BAD_BLOCK_ID 0x1u /* a word's phys_id >= num_pool_blocks (block skipped) */
#define LAZY_DEV_POS_RANGE 0x2u    /* |rotation offset| >= LAZY_MAX_ROPE_OFFSET (offset clamped) */
#define LAZY_DEV_TIMEOUT 0x4u      /* a pipeline wait gave up after its limit */
#define LAZY_DEV_LAYOUT 0x8u       /* the device packer met an invalid layout */
#define LAZY_DEV_BAD_LEN 0x10u     /* seq_lens < 0 or > 16*max_blocks_per_seq (clamped) */

/* Largest |offset| the rotation table covers (positions and offsets). */
#define LAZY_MAX_ROPE_OFFSET (1 << 24)

typedef struct {
  int32_t num_seqs;           /* B >= 0 */
  int32_t num_q_heads;        /* Hq; Hq % Hkv == 0; q-head h reads KV head h / (Hq/Hkv) */
  int32_t num_kv_heads;       /* Hkv >= 1 */
  int32_t head_dim;           /* d: 64 or 128 */
  int32_t block_size;         /* must be 16 */
  int32_t num_pool_blocks;    /* rows of k_pool / v_pool, < 2^id_bits */
  int32_t max_blocks_per_seq; /* row stride of block_words */
  int32_t id_bits;            /* 8..24; 0 selects the default 18 */
  int32_t dtype;              /* lazy_dtype of q, pools and out */
  int32_t lazy;               /* 1: rotate on the fly (LazyAttention). 0: control -- the pool
                                 already holds absolute-position K, no per-document rotation */
  double rope_theta;          /* 1e4, 5e5, ... */
  float sm_scale;             /* softmax scale; 0 selects 1/sqrt(head_dim) */
  int32_t num_splits;         /* decode split-K factor; 0 = choose from the shapes and SM count */
  int32_t key_positions;      /* 0: a block word's offset is taken from its document's start p
                                 (RoPE). 1: from the position of the block's first key, so every
                                 key's absolute position is the word's position plus its slot
                                 (ALiBi). The packers write either form; the ALiBi calls require
                                 1, every other attention call and the materialiser require 0
                                 (LAZY_ERR_INVALID_ARG) */
  int32_t kv_dtype;           /* 0: the pools have `dtype`. LAZY_FP8_E4M3: the pools hold one
                                 e4m3 byte per element (same [block][head][16][d] layout), a
                                 key's value is code * k_scale and a value's code * v_scale.
                                 Only lazy_attn_decode (and _noalloc) and lazy_attn_decode_shared
                                 with dtype LAZY_BF16 and head_dim 128 take it; the ALiBi calls,
                                 the prefill and the materialiser return LAZY_ERR_UNSUPPORTED.
                                 Pools 16-byte aligned. */
  float k_scale;              /* FP8 dequantisation scales: finite, > 0; 0 selects 1 */
  float v_scale;
} lazy_attn_params;

/* Human-readable name of a lazy_status value. Never NULL. */
const char *lazy_attn_status_string(int status);

/* ---------------------------------------------------------------- rotation table
 * Per-frequency rotation rates in turns, t_i = w_i / (2 pi), computed in fp64 on
 * the device once per (head_dim, rope_theta) and stored as an unevaluated sum of
 * two fp32 values (hi, lo). For an integer offset n the kernels form n*t_i with
 * an error-free product, drop the whole turns exactly (n*t_i - rint(n*t_i) is
 * exact in fp32), and evaluate cos/sin(2 pi * fraction) with sincospif. The
 * angle error stays below about 5e-7 rad for every |n| < LAZY_MAX_ROPE_OFFSET,
 * with no memory access per offset.
 * A second part holds (cos, sin)(i * w_f) for the row offsets i = 0 .. LAZY_ROPE_ROWS-1
 * of a prefill query tile, also computed in fp64 and rounded to fp32: a tile whose
 * rows sit at base + i gets its angles by angle addition from the tile's base angles
 * (sincospif once per frequency per tile instead of once per row).
 * Layout: float2 [head_dim/2] = (hi, lo), then float2 [LAZY_ROPE_ROWS][head_dim/2] =
 * (cos, sin). Caller-owned device memory of at least lazy_attn_rope_table_bytes(p)
 * bytes, 16-byte aligned; read-only to every other call. */
#define LAZY_ROPE_ROWS 128
size_t lazy_attn_rope_table_bytes(const lazy_attn_params *p);
int lazy_attn_rope_table_init(const lazy_attn_params *p, void *table, size_t table_bytes,
                              lazy_stream_t stream);

/* Frequency scaling of the rotation (not in the pages, which state the method for
 * RoPE in general): the Llama-3.1 rule changes only the frequencies w_f = theta^(-2f/d),
 * so every kernel picks it up from the table. With wavelength lambda = 2 pi / w,
 * lambda_hi = original_max_position / high_freq_factor and lambda_lo =
 * original_max_position / low_freq_factor, a frequency is kept when lambda < lambda_hi,
 * divided by `factor` when lambda > lambda_lo, and otherwise interpolated with
 * s = (original_max_position / lambda - low_freq_factor) / (high_freq_factor - low_freq_factor):
 * w' = (1 - s) w / factor + s w. lazy_attn_rope_table_init_scaled fills the same table
 * as lazy_attn_rope_table_init from the scaled frequencies (scaling NULL: unscaled).
 * Requires factor > 0 and 0 < low_freq_factor < high_freq_factor and
 * original_max_position > 0, else LAZY_ERR_INVALID_ARG.
 * Interleaved (GPT-J) pairing (2f, 2f+1) needs no entry point: it is rotate-half
 * pairing on a head dimension permuted as [0, 2, 4, ..., d-2, 1, 3, ..., d-1]; a
 * caller that applies that permutation to q and to the stored K rows (V and out are
 * not rotated and stay as they are) gets the interleaved results, since one common
 * permutation of q and k leaves every score unchanged. */
typedef struct {
  double factor;
  double low_freq_factor;
  double high_freq_factor;
  int32_t original_max_position;
} lazy_rope_scaling;
int lazy_attn_rope_table_init_scaled(const lazy_attn_params *p, const lazy_rope_scaling *scaling, void *table,
                                     size_t table_bytes, lazy_stream_t stream);

/* Explicit frequencies: fills the same table from freqs_host[head_dim/2], the rate of
 * pair f (dims f and f + head_dim/2) in radians per position, fp64 host memory read
 * during the call. Each rate must be finite with 0 <= w <= 4 (RoPE's fastest rate is
 * 1), else LAZY_ERR_INVALID_ARG. A rate of 0 leaves its pair unrotated, which gives
 * partial rotary (GPT-NeoX / GPT-J rotary_dim: only the first r dims rotate, pairs
 * (f, f + r/2) or (2f, 2f+1) at rates theta^(-2f/r)): permute the head dimension of q
 * and of the stored K rows so that the rotary pairs become pairs (f, f + head_dim/2),
 * f < r/2, and the other dims fill the remaining pairs; pass theta^(-2f/r) for f < r/2
 * and 0 beyond. V and out keep their order. Other frequency rules (NTK-aware or YaRN
 * interpolation, whose temperature is sm_scale) are rate vectors too. */
int lazy_attn_rope_table_init_freqs(const lazy_attn_params *p, const double *freqs_host, void *table,
                                    size_t table_bytes, lazy_stream_t stream);

/* Host helper for the layout above: for a head of head_dim dims whose first rot_dims
 * rotate (rot_dims even, 2 <= rot_dims <= head_dim; rot_dims = head_dim is full
 * rotary) with rotate-half pairs (f, f + rot_dims/2), or interleaved pairs (2f, 2f+1)
 * when `interleaved`, writes perm_out[head_dim] (new dim i holds old dim perm_out[i])
 * and freqs_out[head_dim/2] (theta^(-2f/rot_dims) for f < rot_dims/2, then 0).
 * Returns LAZY_ERR_INVALID_ARG on bad sizes. */
int lazy_attn_rotary_layout_host(int32_t head_dim, int32_t rot_dims, int32_t interleaved, double theta,
                                 int32_t *perm_out, double *freqs_out);

/* ---------------------------------------------------------------- block-word packer
 * Builds block_words and seq_lens from per-sequence document lists (CSR):
 *   seg_indptr [B+1]; segment k of sequence s (seg_indptr[s] <= k < seg_indptr[s+1])
 *   uses the first seg_len[k] >= 1 tokens of document seg_doc[k];
 *   seq_pos0 [B] (may be NULL = all 0): global position of the sequence's first
 *   token; segment k starts at p_k = seq_pos0[s] + sum of earlier seg_len;
 *   doc_block_indptr [num_docs+1], doc_blocks: physical block ids of each
 *   document in token order.
 * Words past a sequence's last block are written as 0.
 *
 * Host form: every array is host memory; validates and packs on the host. Returns
 * LAZY_ERR_LAYOUT on a segment longer than its document, a block id outside the
 * pool or id field, an offset that does not fit, or more than max_blocks_per_seq
 * blocks in a sequence. */
int lazy_attn_pack_block_words_host(const lazy_attn_params *p, int32_t num_docs, const int32_t *seg_indptr_host,
                                    const int32_t *seg_doc_host, const int32_t *seg_len_host,
                                    const int32_t *seq_pos0_host, const int32_t *doc_block_indptr_host,
                                    const int32_t *doc_blocks_host, uint32_t *block_words_host,
                                    int32_t *seq_lens_host);

/* Device form: every array is device memory (seq_pos0 may be NULL); one warp per
 * sequence packs on the GPU. Layout errors set LAZY_DEV_LAYOUT in the status word
 * and write seq_lens[s] = 0 for the offending sequence. Same output bits as the
 * host form. */
int lazy_attn_pack_block_words(const lazy_attn_params *p, int32_t num_docs, const int32_t *seg_indptr,
                               const int32_t *seg_doc, const int32_t *seg_len, const int32_t *seq_pos0,
                               const int32_t *doc_block_indptr, const int32_t *doc_blocks,
                               uint32_t *block_words, int32_t *seq_lens, lazy_stream_t stream);

/* ---------------------------------------------------------------- decode
 * One query per sequence ("Implementação Técnica", item 2, Decoding: query tile
 * M = 1; the query is re-rotated only when the relative offset changes, i.e. at
 * a new document; memory traffic is K and V only).
 *   q       [B][Hq][d] dtype, UNROTATED
 *   q_pos   [B] int32 absolute position m of each query; every cached key must
 *           sit at a position <= m (all keys in the table are attended to)
 *   out     [B][Hq][d] dtype: softmax(<R_{m-p} q, K_stored> * sm_scale) V
 *           (zero for a sequence with seq_lens == 0)
 *   workspace: device scratch for split-K partials, at least
 *           lazy_attn_decode_workspace_bytes(p) bytes (0 when one split suffices),
 *           256-byte aligned; not read before it is written.
 * lazy == 0 (control): q is rotated once by R_m and the pool is read as already
 * holding absolute-position keys. */
size_t lazy_attn_decode_workspace_bytes(const lazy_attn_params *p);
int lazy_attn_decode(const lazy_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                     const uint32_t *block_words, const int32_t *seq_lens, const int32_t *q_pos,
                     const void *rope_table, void *out, void *workspace, size_t workspace_bytes,
                     lazy_stream_t stream);

/* ---------------------------------------------------------------- shared-run decode
 * The same decode result as lazy_attn_decode, for batches whose sequences cite
 * the same cached documents. Because stored keys carry no global position
 * ("Metodologia: Codificação Posicional Diferida"), one physical block serves
 * every sequence that cites it, at whatever offset each places it; this entry
 * point reads each such block once per KV head for the whole batch instead of
 * once per sequence, and applies each sequence's own relative rotation R_{m-p}
 * to its query ("Implementação Técnica", item 2: one rotation per document run).
 *
 * Plan (host): lazy_attn_plan_shared_host takes the document lists of the
 * block-word packer (same arguments, host memory). Occurrences of one document
 * with the same used length read the same physical blocks; they are grouped,
 * split into sets of at most LAZY_PLAN_MAX_MEMBERS members and at most R query
 * rows (members x query heads per KV head), and each set's blocks are cut into
 * chunks of chunk_blocks logical blocks. R is 128 when a KV head serves at least
 * 8 query heads, head_dim is 128 and the pools are not e4m3 (the decode then runs
 * on the 5th-generation tensor cores, one 128-row tile per item), else 64 (plan
 * with the kv_dtype the decode will use). chunk_blocks 0 selects 32,
 * or, for R = 128, about one item per resident CTA (2 x 152 / num_kv_heads items):
 * the sets' blocks summed, divided by that count, rounded up to a multiple of 4
 * and kept within 32 .. 256. It writes
 *   items_host [num_items][LAZY_PLAN_ITEM_INTS] int32, one work item each:
 *     [0] src_seq, [1] b0, [2] nblk, [3] last_valid, [4] nmem, [5] c0, [6..7] 0:
 *         nblk logical blocks of sequence src_seq from block b0, all full but
 *         the last (last_valid slots), computed for nmem members; they are the
 *         blocks c0 .. c0+nblk-1 of their document (key k of block c0 + i is the
 *         document's key 16 (c0 + i) + k);
 *     [8 + 4j ..] member j < nmem: {seq, b0, slot, 0}: sequence seq holds the
 *         same physical blocks at its logical blocks b0 .. b0+nblk-1 and its
 *         partial result goes to `slot`; unused member entries are 0;
 *     [72 + k] k < min(nblk, LAZY_PLAN_ITEM_BLOCK_IDS): physical id of the
 *         item's block k (what src_seq's block word b0 + k names), 0 beyond: the
 *         kernel starts the loads from these ids and checks them against the
 *         block words (a mismatch sets LAZY_DEV_LAYOUT);
 *   slot_indptr_host [B+1]: the slots of sequence s are slot_indptr[s] ..
 *     slot_indptr[s+1]-1;
 *   counts_host [2] = {num_items, num_slots}.
 * Items are ordered by decreasing block count (ties in the order of first
 * appearance of their document).
 * `capacity` bounds the item count (the number
 * of logical blocks in the batch always suffices). Returns LAZY_ERR_LAYOUT on the
 * packer's layout errors, and LAZY_ERR_WORKSPACE if capacity is too small.
 *
 * Decode: items and slot_indptr copied to device memory unchanged (items 16-byte
 * aligned), block_words packed from the same document lists. workspace: at least
 * lazy_attn_decode_shared_workspace_bytes(p, num_slots) bytes, 16-byte aligned.
 * dtype bf16 only; at most 64 query heads per KV head. kv_dtype LAZY_FP8_E4M3
 * (head_dim 128): pools of e4m3 codes, read as 16-row x 128-byte boxes, on the
 * mma.sync kernel at every ratio (items of at most 64 rows). A member whose first block does
 * not hold the item's physical block, or an item outside the table, sets
 * LAZY_DEV_LAYOUT and is skipped. */
#define LAZY_PLAN_MAX_MEMBERS 16
#define LAZY_PLAN_ITEM_BLOCK_IDS 32
#define LAZY_PLAN_ITEM_INTS (8 + 4 * LAZY_PLAN_MAX_MEMBERS + LAZY_PLAN_ITEM_BLOCK_IDS)
int lazy_attn_plan_shared_host(const lazy_attn_params *p, int32_t num_docs, const int32_t *seg_indptr_host,
                               const int32_t *seg_doc_host, const int32_t *seg_len_host,
                               const int32_t *doc_block_indptr_host, const int32_t *doc_blocks_host,
                               int32_t chunk_blocks, int32_t capacity, int32_t *items_host,
                               int32_t *slot_indptr_host, int32_t *counts_host);
size_t lazy_attn_decode_shared_workspace_bytes(const lazy_attn_params *p, int32_t num_slots);
int lazy_attn_decode_shared(const lazy_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                            const uint32_t *block_words, const int32_t *q_pos, const void *rope_table,
                            int32_t num_items, const int32_t *items, int32_t num_slots, const int32_t *slot_indptr,
                            void *out, void *workspace, size_t workspace_bytes, lazy_stream_t stream);

/* The two halves of lazy_attn_decode_shared as separate calls (same arguments and
 * checks). The split-K decode is two passes: partial results per document chunk,
 * then their merge ("KV Cache, Flash Attention & Otimização de Inferência",
 * "Flash Attention -- tiling": the running-maximum rescale). Keeping the partials
 * lets a caller merge chunks computed elsewhere (another stream, or another GPU's
 * share of the documents, gathered first), or time the two passes apart.
 * lazy_attn_decode_shared_partials runs the work-item kernel only and leaves in
 * `workspace`: fp32 o[num_slots][Hq][head_dim] (unnormalised weighted values, in
 * log2 units of the running maximum), then fp32 (m, l)[num_slots][Hq] (running
 * maximum in log2 units and weight sum; (-inf, 0) for an empty slot).
 * lazy_attn_decode_shared_combine merges each sequence's slots of such a workspace
 * into out [B][Hq][head_dim] bf16: out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k
 * over the slots k of slot_indptr, M = max_k m_k; 0 for a sequence without slots.
 * lazy_attn_decode_shared = partials, then combine (launched so that the combine's
 * start overlaps the work-item kernel's last CTAs). */
int lazy_attn_decode_shared_partials(const lazy_attn_params *p, const void *q, const void *k_pool,
                                     const void *v_pool, const uint32_t *block_words, const int32_t *q_pos,
                                     const void *rope_table, int32_t num_items, const int32_t *items,
                                     int32_t num_slots, void *workspace, size_t workspace_bytes,
                                     lazy_stream_t stream);
int lazy_attn_decode_shared_combine(const lazy_attn_params *p, int32_t num_slots, const int32_t *slot_indptr,
                                    const void *workspace, size_t workspace_bytes, void *out, lazy_stream_t stream);

/* ALiBi ("Resumo Técnico: LazyAttention", "Principais Contribuições", item 4: the
 * mechanism carries over to relative position encodings such as ALiBi): the same
 * calls with every score of query head h also biased by -alibi_slopes[h] * (m - n)
 * before the softmax, for a key at absolute position n and the query at m = q_pos.
 * Stored keys carry no position; n comes from the block words packed with
 * p->key_positions = 1 (a block's word gives the position of its first key; n is
 * that plus the slot), and the bias is formed on the fly. ALiBi models do not rotate
 * q or k: pass a table built by lazy_attn_rope_table_init_freqs from zero rates (the
 * calls do not rotate, whatever p->lazy says). alibi_slopes: device fp32 [Hq], 4-byte
 * aligned; p->key_positions must be 1, else LAZY_ERR_INVALID_ARG. bf16 only. The
 * prefill's ALiBi form, lazy_attn_prefill_alibi, is declared after lazy_attn_prefill. */
int lazy_attn_decode_alibi(const lazy_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                           const uint32_t *block_words, const int32_t *seq_lens, const int32_t *q_pos,
                           const void *rope_table, const float *alibi_slopes, void *out, void *workspace,
                           size_t workspace_bytes, lazy_stream_t stream);
int lazy_attn_decode_shared_alibi(const lazy_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                                  const uint32_t *block_words, const int32_t *q_pos, const void *rope_table,
                                  int32_t num_items, const int32_t *items, int32_t num_slots,
                                  const int32_t *slot_indptr, const float *alibi_slopes, void *out, void *workspace,
                                  size_t workspace_bytes, lazy_stream_t stream);

/* The usual ALiBi slopes for num_heads heads (host, out[num_heads]): 2^(-8 i / n),
 * i = 1..n, when n is a power of two; otherwise the slopes of the largest power of
 * two n' below n, followed by the odd-indexed slopes 2^(-8 (2k+1) / (2 n')) for the
 * remaining heads. LAZY_ERR_INVALID_ARG for num_heads outside 1..4096. */
int lazy_attn_alibi_slopes_host(int32_t num_heads, float *out);

/* ---------------------------------------------------------------- decode without allocation
 * The pages have no counterpart for this entry point; it exists for callers that
 * cannot allocate device memory for a workspace: an engine that has reserved nearly
 * all of HBM for its KV-cache pool, a plugin limited to its host framework's
 * buffers, or a latency-critical step that must not call cudaMalloc (which can
 * synchronise the device).
 * Same inputs, outputs and results as lazy_attn_decode, with no workspace
 * argument: the split-K partials live in a file-scope static device array of
 * LAZY_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds until
 * the process exits. The call allocates and frees nothing.
 *  - Returns LAZY_ERR_WORKSPACE, launching nothing, when the split plan of `p`
 *    needs more than LAZY_NOALLOC_SCRATCH_BYTES (lazy_attn_decode_workspace_bytes
 *    tells the need; setting p->num_splits lower reduces it, and 1 needs none).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture. The address is kept with the unique id of the context it was found
 *    in, and looked up again on the first call after that context changed (after
 *    cudaDeviceReset, or with another context made current); that call too should
 *    come before any stream capture.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other threads) race on it and must be serialised by the caller. */
#define LAZY_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */
int lazy_attn_decode_noalloc(const lazy_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                             const uint32_t *block_words, const int32_t *seq_lens, const int32_t *q_pos,
                             const void *rope_table, void *out, lazy_stream_t stream);

/* ---------------------------------------------------------------- prefill
 * Varlen query chunks ("Implementação Técnica", item 1, Prefilling): chunk s
 * has C_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] query rows at absolute
 * positions q_start[s] + i. Its own K/V must already be in the pool as the
 * LAST document of the sequence (C_s tokens, p = q_start[s]); query row i
 * attends to every key of the earlier documents and to chunk keys j <= i.
 * Q is rotated once by R_m per row; each 16-row K block is rotated once, by
 * R_p of its document (one relative rotation per tile, no unrotate pass).
 *   q            [total_q][Hq][d] bf16, UNROTATED
 *   cu_seqlens_q [B+1] int32 device; q_start [B] int32 device
 *   max_q_len    >= every C_s (sizes the work list); total_q = cu_seqlens_q[B]
 *   out          [total_q][Hq][d] bf16
 *   workspace    at least lazy_attn_prefill_workspace_bytes(p, total_q) bytes,
 *                16-byte aligned (LAZY_ERR_WORKSPACE otherwise). With an even GQA
 *                ratio the kernel runs one persistent CTA per SM, each on an equal
 *                share of the (query tile, head pair, K tile) iterations; a query tile
 *                whose K tiles are shared out among several CTAs is merged through the
 *                workspace (per-row arrival counters, which the call zeroes with one
 *                cudaMemsetAsync on `stream`, and fp32 partial results). Its size
 *                depends only on the SM count. Odd GQA ratios need none (0 bytes).
 *                Calls that overlap on the GPU must not share a workspace.
 * Only LAZY_BF16 with head_dim 128 is supported. */
size_t lazy_attn_prefill_workspace_bytes(const lazy_attn_params *p, int32_t total_q);
int lazy_attn_prefill(const lazy_attn_params *p, const void *q, const int32_t *cu_seqlens_q,
                      const int32_t *q_start, int32_t total_q, int32_t max_q_len, const void *k_pool,
                      const void *v_pool, const uint32_t *block_words, const int32_t *seq_lens,
                      const void *rope_table, void *out, void *workspace, size_t workspace_bytes,
                      lazy_stream_t stream);

/* ALiBi prefill ("Resumo Técnico: LazyAttention", "Principais Contribuições", item 4):
 * the same call with every score of query head h biased by
 * -alibi_slopes[h] * (m_i - n) before the softmax, for query row i at m_i =
 * q_start[s] + i and a key at absolute position n (the chunk's own keys included).
 * The block words must be packed with p->key_positions = 1 (a block's word gives the
 * position of its first key; n is that plus the slot) and the rope table built from
 * zero rates (ALiBi models do not rotate; the call never rotates K, and rotates Q
 * only by that table). alibi_slopes: device fp32 [Hq], 4-byte aligned. Both prefill
 * kernels take it (every GQA ratio, MHA included). LAZY_ERR_INVALID_ARG without
 * slopes or with p->key_positions = 0; lazy_attn_prefill refuses key-position words. */
int lazy_attn_prefill_alibi(const lazy_attn_params *p, const void *q, const int32_t *cu_seqlens_q,
                            const int32_t *q_start, int32_t total_q, int32_t max_q_len, const void *k_pool,
                            const void *v_pool, const uint32_t *block_words, const int32_t *seq_lens,
                            const void *rope_table, const float *alibi_slopes, void *out, void *workspace,
                            size_t workspace_bytes, lazy_stream_t stream);

/* ---------------------------------------------------------------- one launch for a mixed batch
 * A continuous-batching step ("KV Cache, Flash Attention & Otimização de Inferência",
 * "Continuous batching": new requests' prompts are prefilled in the same step as the
 * running sequences' decode) as ONE kernel launch: the shared-run decode of a batch
 * (p_dec, its plan and inputs, as lazy_attn_decode_shared takes them) and the
 * prefill of other sequences' chunks (p_pf and the inputs of lazy_attn_prefill),
 * over the same pools and rotation table. The prefill kernel's persistent pipeline
 * also runs the decode's work items: each item is a one-tile unit (member x query
 * head rows, each member rotated by R_{m-p} from its own block word, K used as
 * stored), dealt round robin to the CTAs before their share of the prefill, and the
 * launch ends by merging every decode sequence's partials (the combine of
 * lazy_attn_decode_shared) once its items are done; the launch is cooperative (one
 * CTA per SM, all resident), so that wait always ends.
 * Requirements: dtype bf16, head_dim 128, the same heads, pool, id_bits, sm_scale
 * and lazy = 1 in both params, query heads per KV head a multiple of 16 (the
 * decode's 128-row tensor-core items, plan with p_dec, whose 16-row groups each
 * hold one member's heads); p_dec->kv_dtype and
 * key_positions 0 (LAZY_ERR_UNSUPPORTED otherwise). workspace: at least
 * lazy_attn_mixed_workspace_bytes bytes, 256-byte aligned (the prefill's merge
 * area, the decode partials, one counter per decode sequence; the call zeroes the
 * counters with cudaMemsetAsync on `stream`). A batch with no prefill rows (or no
 * decode sequence) runs as the plain call of the other kind. */
size_t lazy_attn_mixed_workspace_bytes(const lazy_attn_params *p_dec, const lazy_attn_params *p_pf,
                                       int32_t num_slots);
int lazy_attn_mixed(const lazy_attn_params *p_dec, const void *q_dec, const uint32_t *block_words_dec,
                    const int32_t *q_pos, int32_t num_items, const int32_t *items, int32_t num_slots,
                    const int32_t *slot_indptr, void *out_dec, const lazy_attn_params *p_pf, const void *q_pf,
                    const int32_t *cu_seqlens_q, const int32_t *q_start, int32_t total_q, int32_t max_q_len,
                    const uint32_t *block_words_pf, const int32_t *seq_lens_pf, void *out_pf, const void *k_pool,
                    const void *v_pool, const void *rope_table, void *workspace, size_t workspace_bytes,
                    lazy_stream_t stream);

/* ---------------------------------------------------------------- eager materialisation (baseline)
 * The alternative the lazy method avoids ("Declaração do Problema"): a reused
 * document's keys re-rotated to their absolute positions and copied per sequence.
 * For every sequence s and logical block b < ceil(seq_lens[s]/16), writes block
 * s*max_blocks_per_seq + b of k_out / v_out with K rotated by R_p (p of block b's
 * document: R_p R_j k = R_{p+j} k) and V copied, and block_words_out[s][b] with that
 * id and the same offset field (0 for b past the sequence). lazy_attn_decode with
 * lazy = 0 on (k_out, v_out, block_words_out, seq_lens) then computes the same
 * attention without per-document rotation and without any block shared.
 *   k_out, v_out   [num_seqs * max_blocks_per_seq][Hkv][16][d] bf16
 *   block_words_out [num_seqs][max_blocks_per_seq]
 * Needs num_seqs * max_blocks_per_seq <= 2^id_bits (LAZY_ERR_LAYOUT otherwise).
 * bf16 only. */
int lazy_attn_materialize(const lazy_attn_params *p, const void *k_pool, const void *v_pool,
                          const uint32_t *block_words, const int32_t *seq_lens, const void *rope_table, void *k_out,
                          void *v_out, uint32_t *block_words_out, lazy_stream_t stream);

/* ---------------------------------------------------------------- test support
 * Copies every logical K/V slot of every sequence through the decode kernel's
 * own load path (word decode, TMA block loads, hole rule) into dense buffers:
 *   k_out, v_out [B][Hkv][16*max_blocks_per_seq][d] dtype; slot t of logical
 *   block b lands at row 16*b + t; slots that are not valid (holes, past
 *   seq_lens) are written as 0.
 *   pos_out [B][16*max_blocks_per_seq] int32: the absolute position of each
 *   valid slot's token, -1 for invalid slots (may be NULL). */
int lazy_attn_debug_gather(const lazy_attn_params *p, const void *k_pool, const void *v_pool,
                           const uint32_t *block_words, const int32_t *seq_lens, void *k_out, void *v_out,
                           int32_t *pos_out, lazy_stream_t stream);

/* Failure-path test of the bounded waits: lazy_attn_debug_gather (bf16 pools) with
 * the TMA copies of logical block `withhold_block` of sequence 0, KV head 0 never
 * issued, and every pipeline wait of the launch limited to wait_limit_us
 * microseconds (1 .. 2,000,000) instead of 2 s. The withheld block's stage never
 * completes and no copy of it is in flight: the copying warp's wait runs out, sets
 * LAZY_DEV_TIMEOUT and stops; the loading warp's next wait on that stage runs out
 * too, it waits (bounded) for the copies it did issue, and the CTA exits. Other
 * (sequence, head) pairs are gathered as usual. The call returns LAZY_OK after the
 * launch; read the status word to see the timeout. LAZY_ERR_INVALID_ARG for
 * withhold_block < 0 or a limit outside the range, LAZY_ERR_UNSUPPORTED for fp32. */
int lazy_attn_debug_gather_withheld(const lazy_attn_params *p, const void *k_pool, const void *v_pool,
                                    const uint32_t *block_words, const int32_t *seq_lens, void *k_out, void *v_out,
                                    int32_t *pos_out, int32_t withhold_block, uint32_t wait_limit_us,
                                    lazy_stream_t stream);

/* Evaluates the kernels' rotation for n offsets: cs_out[k][i] = (cos, sin) of
 * deltas[k] * w_i, i < head_dim/2, with the device function the attention
 * kernels use. deltas [n] int32 device; cs_out [n][head_dim/2] float2 device. */
int lazy_attn_debug_rope(const lazy_attn_params *p, const void *rope_table, const int32_t *deltas, int32_t n,
                         void *cs_out, lazy_stream_t stream);

/* Reads (and, if clear != 0, zeroes) the current device's status word. Waits for
 * all work on the device first. Returns LAZY_OK, or LAZY_ERR_CUDA. */
int lazy_attn_device_status(uint32_t *flags_out, int clear);

/* Number of kernel launches the library has issued in this process (all devices);
 * lets a caller count GPU work done inside a timed region. */
uint64_t lazy_attn_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* LAZY_ATTN_H_ */
