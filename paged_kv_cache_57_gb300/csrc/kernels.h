// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lazy_attn.h"

namespace lazy {

// Raises a kernel's dynamic shared-memory limit once per device (the attribute
// persists for the process), instead of on every launch.
template <auto Kern>
inline cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}


struct DecodeArgs {
  const void* q;             // [B][Hq][D] unrotated
  const uint32_t* words;     // [B][max_blocks]
  const int32_t* seq_lens;   // [B]
  const int32_t* q_pos;      // [B]
  const float2* rope;        // rotation table: per-frequency turns (hi, lo)
  const void* k_pool;        // [NB][Hkv][16][D] (plain-load kernels)
  const void* v_pool;
  void* out;                 // [B][Hq][D]
  float* ws_o;               // [B][Hq][splits][D]
  float* ws_ml;              // [B][Hq][splits][2]  (running max in log2 units, denominator)
  unsigned int* status;      // device status word
  int B, Hq, Hkv, G, D, max_blocks, id_bits, num_pool_blocks;
  int splits, bps;           // split-K factor and logical blocks per split
  float scale_log2;          // softmax scale * log2(e)
};
// The ALiBi variants' arguments (a separate type keeps the other kernels' argument
// block unchanged).
struct DecodeAlibiArgs : DecodeArgs {
  const float* alibi;  // [Hq] slopes
};

// FP8-KV decode: pools hold e4m3 codes; a key's value is code * k_scale, a value
// row's code * v_scale.
struct DecodeFp8Args : DecodeArgs {
  float k_scale, v_scale;
};

struct GatherArgs {
  const uint32_t* words;
  const int32_t* seq_lens;
  const void* k_pool;
  const void* v_pool;
  void* k_out;               // [B][Hkv][16*max_blocks][D]
  void* v_out;
  int32_t* pos_out;          // [B][16*max_blocks] or null
  unsigned int* status;
  int B, Hkv, D, max_blocks, id_bits, num_pool_blocks;
  // Failure-path test only: logical block `withhold_block` of sequence 0, KV head 0
  // is never loaded (-1: none), and every wait gives up after wait_ns.
  int withhold_block;
  uint64_t wait_ns;
};

struct PackArgs {
  const int32_t* seg_indptr;
  const int32_t* seg_doc;
  const int32_t* seg_len;
  const int32_t* seq_pos0;   // may be null
  const int32_t* doc_block_indptr;
  const int32_t* doc_blocks;
  uint32_t* words;
  int32_t* seq_lens;
  unsigned int* status;
  int B, num_docs, max_blocks, id_bits, num_pool_blocks;
  int key_positions;         // offsets from each block's first key instead of its document's start
};

struct PrefillArgs {
  const int32_t* cu_seqlens_q;
  const int32_t* q_start;
  const uint32_t* words;
  const int32_t* seq_lens;
  const float2* rope;
  void* out;                 // [total_q][Hq][D] bf16
  unsigned int* status;
  int B, Hq, Hkv, G, D, total_q, max_q_len, max_blocks, id_bits, num_pool_blocks;
  int T;                     // query tiles per sequence: ceil(max_q_len / 128)
  float scale_log2;
  // Persistent (stream-K) kernel only: per-row arrival counters of split units,
  // [grid + 1][2][128], zeroed before each launch; fp32 partials [2 * grid][2][128][132].
  int* counters;
  float* partials;
};
// ALiBi prefill: no rotation (key-position words), score of query head h and a key
// at position n biased by slope_h (n - m) for the query at m.
struct PrefillAlibiArgs : PrefillArgs {
  const float* alibi;  // [Hq] slopes
};
// One launch for a continuous batch (prefill_stream.cu): the stream-K prefill kernel
// also runs the shared-run decode's work items, as one-tile units of its pipeline,
// and merges each decode sequence's partials at its end.
struct MixedArgs : PrefillArgs {
  const void* q_dec;           // [B_dec][Hq][D] unrotated
  const uint32_t* words_dec;   // [B_dec][max_blocks_dec]
  const int32_t* q_pos;        // [B_dec]
  const int32_t* items;        // the shared-run plan's items
  const int32_t* slot_indptr;  // [B_dec + 1]
  void* out_dec;               // [B_dec][Hq][D] bf16
  float* ws_o;                 // [num_slots][Hq][D] decode partials
  float* ws_ml;                // [num_slots][Hq][2]
  int* seq_done;               // [B_dec] decode units finished per sequence (zeroed before the launch)
  int B_dec, max_blocks_dec, num_items, num_slots;
};
constexpr int PREFILL_PARTIAL_ROW_FLOATS = 128 + 4;
constexpr int pf_tile_rows = 128;  // query rows per prefill tile

// Shared-run decode (decode_shared.cu): one CTA per (work item, KV head).
struct SharedDecodeArgs {
  const void* q;             // [B][Hq][D] unrotated
  const uint32_t* words;     // [B][max_blocks]
  const int32_t* q_pos;      // [B]
  const float2* rope;        // rotation table
  const int32_t* items;      // [num_items][LAZY_PLAN_ITEM_INTS]: header, then members {seq, first block, slot}
  const int32_t* slot_indptr;  // [B+1]
  void* out;                 // [B][Hq][D] bf16
  float* ws_o;               // [num_slots][Hq][D]
  float* ws_ml;              // [num_slots][Hq][2]
  unsigned int* status;
  int B, Hq, Hkv, G, D, max_blocks, id_bits, num_pool_blocks;
  int num_items, num_slots;
  float scale_log2;
};
// The ALiBi variants' arguments: the same and the slopes. (A separate type keeps the
// other kernels' argument block, and so their register allocation, unchanged.)
struct SharedAlibiArgs : SharedDecodeArgs {
  const float* alibi;  // [Hq] slopes
};

// FP8 (e4m3) pools on the shared-run decode: keys code * k_scale, values code * v_scale.
struct SharedFp8Args : SharedDecodeArgs {
  float k_scale, v_scale;
};

// Eager materialisation (materialize.cu): per-sequence copies with K at absolute positions.
struct MaterializeArgs {
  const void* k_pool;        // [NB][Hkv][16][D]
  const void* v_pool;
  const uint32_t* words;     // [B][max_blocks]
  const int32_t* seq_lens;   // [B]
  const float2* rope;        // rotation table
  void* k_out;               // [B * max_blocks][Hkv][16][D]
  void* v_out;
  uint32_t* words_out;       // [B][max_blocks]
  unsigned int* status;
  int B, Hkv, D, max_blocks, id_bits, num_pool_blocks;
};
cudaError_t launch_materialize(const MaterializeArgs& a, cudaStream_t st);

// Query rows per shared-run work item: 128 where the tensor-core kernel
// (decode_shared_tc.cu) serves the call -- at least 8 query heads per KV head and
// D = 128 -- else 64 (decode_shared.cu). The planner and the decode call both
// follow it. (Measured: at 8 query heads per KV head, items of 16 members on the
// tensor cores beat items of 8 on mma.sync; at 4, 16-member items fill only half
// a tile and mma.sync stays ahead.)
inline int shared_rows_cap(int G, int D) { return (G >= 8 && D == 128) ? 128 : 64; }
// Resident CTAs of the tensor-core kernel on a GB300 (2 per SM x 152 SMs): its
// automatic chunk length aims at about this many CTAs, so that each CTA's fixed
// cost (record, query rotation, partials) is paid as few times as the machine allows.
constexpr int kSharedTcSlots = 2 * 152;

// Host planner of the shared-run decode (shared_plan.cu). counts = {items, slots}.
// chunk_blocks <= 0 picks the chunk from the batch: about auto_items items in all,
// 32 to 256 blocks in multiples of 4. Items run longest first; with spread_small,
// items of at most 8 blocks are spread evenly through the order instead.
int plan_shared_host(int B, int G, int rows_cap, int max_blocks, int num_pool_blocks, int num_docs, const int32_t* seg_indptr,
                     const int32_t* seg_doc, const int32_t* seg_len, const int32_t* doc_block_indptr,
                     const int32_t* doc_blocks, int chunk_blocks, int auto_items, int capacity, int32_t* items,
                     int32_t* slot_indptr, int32_t* counts, bool spread_small = false);

// Every launcher returns the cudaError_t of its launch.
// explicit_w (host, head_dim/2 rates in radians per position) overrides theta and scaling.
cudaError_t launch_rope_table(float2* table, int head_dim, double theta, const lazy_rope_scaling* scaling,
                              const double* explicit_w, cudaStream_t st);
cudaError_t launch_debug_rope(const float2* table, const int32_t* deltas, int n, int head_dim, float2* out,
                              unsigned int* status, cudaStream_t st);
cudaError_t launch_pack(const PackArgs& a, cudaStream_t st);
cudaError_t launch_decode_f32(const DecodeArgs& a, bool lazy, cudaStream_t st);
// alibi: null, or [Hq] ALiBi slopes (key-position words; no rotation).
cudaError_t launch_decode_bf16(const DecodeArgs& a, const float* alibi, bool lazy, const CUtensorMap& kmap,
                               const CUtensorMap& vmap,
                               cudaStream_t st);
// FP8-KV form of launch_decode_bf16 (D = 128): kmap / vmap are e4m3 [rows][128] maps
// with 16-row x 128-byte boxes.
cudaError_t launch_decode_fp8(const DecodeArgs& a, float k_scale, float v_scale, bool lazy, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t st);
cudaError_t launch_combine(const DecodeArgs& a, bool out_bf16, cudaStream_t st);
cudaError_t launch_gather_bf16(const GatherArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t st);
cudaError_t launch_gather_f32(const GatherArgs& a, cudaStream_t st);
// Chooses the prefill kernel: the stream-K two-tile kernel for even GQA ratios (it
// needs a.counters / a.partials and `grid` = prefill_stream_grid()), else the
// TMEM-Q one-tile kernel.
cudaError_t launch_prefill(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int grid, cudaStream_t st, const float* alibi = nullptr);
// Two query tiles per CTA, one CTA per SM, stream-K over (unit, K tile); even GQA ratio.
cudaError_t launch_prefill_stream(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int grid, cudaStream_t st, const float* alibi = nullptr);
cudaError_t launch_mixed(const MixedArgs& a, const CUtensorMap& qmap, const CUtensorMap& qmap_dec,
                         const CUtensorMap& kmap, const CUtensorMap& vmap, int grid, cudaStream_t st);
size_t prefill_stream_workspace_bytes(int grid);  // counters, then partials
size_t prefill_stream_counter_bytes(int grid);
int prefill_stream_grid();

// One query tile per CTA with the rotated Q tile in tensor memory; any GQA ratio.
cudaError_t launch_prefill_tq(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t st, const float* alibi = nullptr);

// alibi: null, or [Hq] ALiBi slopes (lazy mode only).
cudaError_t launch_decode_shared(const SharedDecodeArgs& a, const float* alibi, bool lazy, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t st);
// The same kernel on e4m3 pools (d = 128; every query-head count up to 64 per KV head,
// items of at most 64 rows).
cudaError_t launch_decode_shared_fp8(const SharedDecodeArgs& a, float k_scale, float v_scale, bool lazy,
                                     const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st);
cudaError_t launch_decode_shared_tc(const SharedDecodeArgs& a, const float* alibi, bool lazy,
                                    const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st);
cudaError_t launch_shared_combine(const SharedDecodeArgs& a, cudaStream_t st);

// Shared-memory bytes a bf16 decode CTA needs (for occupancy-based split planning).
int decode_bf16_smem_bytes(int D, int G);

}  // namespace lazy
