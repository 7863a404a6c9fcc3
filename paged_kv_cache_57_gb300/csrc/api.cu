// api.cu -- the C ABI declared in include/lazy_attn.h: argument checks, host-side
// block-word packing, tensor-map encoding, split planning and kernel launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

// The per-device status word (one copy per device the library is loaded on).
__device__ unsigned int g_lazy_status = 0u;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultIdBits = 18;
constexpr int kDefaultSmCount = 152;  // used only when no device is visible (size queries)

std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct Checked {
  int id_bits = kDefaultIdBits;
  int G = 1;
};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

unsigned int* status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lazy_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_status_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return kDefaultSmCount;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kDefaultSmCount;
    }
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

bool encoder_ready() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// cuTensorMapEncodeTiled through a small per-thread cache of the last maps made
// (bf16, 128-byte swizzle, no interleave, L2 promotion 256 B, no fill): a call with
// the same pool pointers and shapes as a recent one reuses its maps.
static bool encode_cached(CUtensorMap* m, cuuint32_t rank, const void* base, const cuuint64_t* dims,
                          const cuuint64_t* strides, const cuuint32_t* box,
                          CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  struct Entry {
    const void* base;
    CUtensorMapDataType dtype;
    cuuint32_t rank;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    CUtensorMap map;
    bool valid;
  };
  thread_local Entry cache[8] = {};
  thread_local int next = 0;
  Entry key{};
  key.base = base;
  key.dtype = dtype;
  key.rank = rank;
  for (cuuint32_t i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides[i];
  }
  for (Entry& e : cache)
    if (e.valid && e.base == key.base && e.dtype == key.dtype && e.rank == key.rank && std::memcmp(e.dims, key.dims, sizeof(key.dims)) == 0 &&
        std::memcmp(e.strides, key.strides, sizeof(key.strides)) == 0 &&
        std::memcmp(e.box, key.box, sizeof(key.box)) == 0) {
      *m = e.map;
      return true;
    }
  if (!encoder_ready()) return false;
  cuuint32_t es[3] = {1, 1, 1};
  if (g_encode(m, dtype, rank, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  key.map = *m;
  key.valid = true;
  cache[next] = key;
  next = (next + 1) % 8;
  return true;
}

// 2-D bf16 view [rows][d] with 16-row x 64-column boxes, 128-byte swizzle.
bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, int d, uint32_t box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, box_rows};
  return encode_cached(m, 2, base, dims, strides, box);
}

// 2-D e4m3 view [rows][128] with 16-row x 128-byte boxes, 128-byte swizzle.
bool encode_rows_map_fp8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  return encode_cached(m, 2, base, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// 3-D bf16 view of the same [rows][d] pool as (column in a 64-column half, row, half):
// one box of 64 columns x box_rows rows x d/64 halves lands as the d/64 swizzled
// 64-column boxes of encode_rows_map placed one after the other, in one copy.
bool encode_block_map(CUtensorMap* m, const void* base, uint64_t rows, int d, uint32_t box_rows) {
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(d / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, 128};
  cuuint32_t box[3] = {64, box_rows, (cuuint32_t)(d / 64)};
  return encode_cached(m, 3, base, dims, strides, box);
}

// 3-D bf16 view of q [total_q][Hq][d]: boxes of 64 columns x 1 head x box_rows rows.
bool encode_q_map(CUtensorMap* m, const void* base, uint64_t total_q, int hq, int d, uint32_t box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  return encode_cached(m, 3, base, dims, strides, box);
}

// Decode queries [B][Hq][d] for the mixed launch: box = 64 columns x g heads x 1 sequence.
bool encode_dec_q_map(CUtensorMap* m, const void* base, uint64_t B, int hq, int d, int g) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)g, 1};
  return encode_cached(m, 3, base, dims, strides, box);
}

// The pools hold e4m3 codes (FP8 KV; only the per-sequence decode reads them).
static bool kv_fp8(const lazy_attn_params* p) { return p->kv_dtype == LAZY_FP8_E4M3 && p->dtype != LAZY_FP8_E4M3; }

int check_params(const lazy_attn_params* p, Checked* c) {
  if (!p) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads != 0)
    return LAZY_ERR_INVALID_ARG;
  if (p->num_pool_blocks < 0 || p->max_blocks_per_seq < 0 || p->max_blocks_per_seq > (1 << 26))
    return LAZY_ERR_INVALID_ARG;
  if (p->block_size != lazy::kBlock) return LAZY_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return LAZY_ERR_UNSUPPORTED;
  if (p->dtype != LAZY_F32 && p->dtype != LAZY_BF16) return LAZY_ERR_UNSUPPORTED;
  if (p->lazy != 0 && p->lazy != 1) return LAZY_ERR_INVALID_ARG;
  if (!(p->rope_theta > 0.0) || !std::isfinite(p->rope_theta)) return LAZY_ERR_INVALID_ARG;
  if (!(p->sm_scale >= 0.f) || !std::isfinite(p->sm_scale)) return LAZY_ERR_INVALID_ARG;
  if (p->num_splits < 0) return LAZY_ERR_INVALID_ARG;
  if (p->key_positions != 0 && p->key_positions != 1) return LAZY_ERR_INVALID_ARG;
  if (p->kv_dtype != 0 && p->kv_dtype != p->dtype && p->kv_dtype != LAZY_FP8_E4M3) return LAZY_ERR_UNSUPPORTED;
  if (!(p->k_scale >= 0.f) || !std::isfinite(p->k_scale) || !(p->v_scale >= 0.f) || !std::isfinite(p->v_scale))
    return LAZY_ERR_INVALID_ARG;
  c->id_bits = p->id_bits ? p->id_bits : kDefaultIdBits;
  if (c->id_bits < 8 || c->id_bits > 24) return LAZY_ERR_INVALID_ARG;
  if ((int64_t)p->num_pool_blocks > ((int64_t)1 << c->id_bits)) return LAZY_ERR_INVALID_ARG;
  c->G = p->num_q_heads / p->num_kv_heads;
  return LAZY_OK;
}

float scale_log2(const lazy_attn_params* p) {
  const double s = p->sm_scale > 0.f ? (double)p->sm_scale : 1.0 / std::sqrt((double)p->head_dim);
  return (float)(s * 1.4426950408889634);  // log2(e)
}

// Split-K plan: about four waves of two CTAs per SM, at least 16 blocks per split.
void plan_splits(const lazy_attn_params* p, int* splits, int* bps) {
  const int mb = p->max_blocks_per_seq > 0 ? p->max_blocks_per_seq : 1;
  int s = p->num_splits;
  if (s <= 0) {
    const int64_t units = (int64_t)(p->num_seqs > 0 ? p->num_seqs : 1) * p->num_kv_heads;
    const int64_t target = (int64_t)sm_count() * 2 * 4;
    s = (int)((target + units - 1) / units);
    const int max_s = mb / 16 > 1 ? mb / 16 : 1;
    s = s < max_s ? s : max_s;
  }
  s = s < 1 ? 1 : (s > mb ? mb : s);
  *bps = (mb + s - 1) / s;
  *splits = (mb + *bps - 1) / *bps;
}

size_t decode_ws_bytes(const lazy_attn_params* p, int splits) {
  if (splits <= 1) return 0;
  const size_t parts = (size_t)p->num_seqs * p->num_q_heads * splits;
  return parts * p->head_dim * sizeof(float) + parts * 2 * sizeof(float);
}

int launched(cudaError_t e) {
  if (e != cudaSuccess) return LAZY_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return LAZY_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

extern "C" {

const char* lazy_attn_status_string(int status) {
  switch (status) {
    case LAZY_OK: return "LAZY_OK";
    case LAZY_ERR_INVALID_ARG: return "LAZY_ERR_INVALID_ARG: invalid argument";
    case LAZY_ERR_UNSUPPORTED: return "LAZY_ERR_UNSUPPORTED: shape or dtype not supported";
    case LAZY_ERR_WORKSPACE: return "LAZY_ERR_WORKSPACE: workspace or table too small or misaligned";
    case LAZY_ERR_LAYOUT: return "LAZY_ERR_LAYOUT: documents and blocks do not form a valid block table";
    case LAZY_ERR_CUDA: return "LAZY_ERR_CUDA: a CUDA call or launch failed";
    case LAZY_ERR_DEVICE: return "LAZY_ERR_DEVICE: the device status word reported a fault";
    default: return "unknown lazy_attn status";
  }
}

uint64_t lazy_attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t lazy_attn_rope_table_bytes(const lazy_attn_params* p) {
  Checked c;
  if (check_params(p, &c) != LAZY_OK) return 0;
  return (size_t)(p->head_dim / 2) * (1 + LAZY_ROPE_ROWS) * sizeof(float2);
}

int lazy_attn_rope_table_init(const lazy_attn_params* p, void* table, size_t table_bytes, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (!table) return LAZY_ERR_INVALID_ARG;
  if (table_bytes < lazy_attn_rope_table_bytes(p) || !aligned16(table)) return LAZY_ERR_WORKSPACE;
  return launched(lazy::launch_rope_table(static_cast<float2*>(table), p->head_dim, p->rope_theta, nullptr, nullptr,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int lazy_attn_rope_table_init_scaled(const lazy_attn_params* p, const lazy_rope_scaling* scaling, void* table,
                                     size_t table_bytes, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (!table) return LAZY_ERR_INVALID_ARG;
  if (scaling && !(scaling->factor > 0.0 && scaling->low_freq_factor > 0.0 &&
                   scaling->high_freq_factor > scaling->low_freq_factor && scaling->original_max_position > 0))
    return LAZY_ERR_INVALID_ARG;
  if (table_bytes < lazy_attn_rope_table_bytes(p) || !aligned16(table)) return LAZY_ERR_WORKSPACE;
  return launched(lazy::launch_rope_table(static_cast<float2*>(table), p->head_dim, p->rope_theta, scaling, nullptr,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int lazy_attn_rotary_layout_host(int32_t head_dim, int32_t rot_dims, int32_t interleaved, double theta,
                                 int32_t* perm_out, double* freqs_out) {
  if (head_dim < 2 || head_dim % 2 || rot_dims < 2 || rot_dims % 2 || rot_dims > head_dim || !(theta > 1.0) ||
      !perm_out || !freqs_out)
    return LAZY_ERR_INVALID_ARG;
  const int h = head_dim / 2, hr = rot_dims / 2, hn = (head_dim - rot_dims) / 2;
  for (int f = 0; f < hr; ++f) {  // rotary pair f -> new dims (f, f + h)
    perm_out[f] = interleaved ? 2 * f : f;
    perm_out[f + h] = interleaved ? 2 * f + 1 : f + hr;
    freqs_out[f] = std::pow(theta, -2.0 * (double)f / (double)rot_dims);
  }
  for (int k = 0; k < hn; ++k) {  // unrotated dims fill the remaining pairs, rate 0
    perm_out[hr + k] = rot_dims + k;
    perm_out[hr + k + h] = rot_dims + hn + k;
    freqs_out[hr + k] = 0.0;
  }
  return LAZY_OK;
}

int lazy_attn_rope_table_init_freqs(const lazy_attn_params* p, const double* freqs_host, void* table,
                                    size_t table_bytes, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (!freqs_host || !table) return LAZY_ERR_INVALID_ARG;
  for (int f = 0; f < p->head_dim / 2; ++f)
    if (!(freqs_host[f] >= 0.0 && freqs_host[f] <= 4.0)) return LAZY_ERR_INVALID_ARG;  // also rejects NaN
  if (table_bytes < lazy_attn_rope_table_bytes(p) || !aligned16(table)) return LAZY_ERR_WORKSPACE;
  return launched(lazy::launch_rope_table(static_cast<float2*>(table), p->head_dim, p->rope_theta, nullptr,
                                          freqs_host, reinterpret_cast<cudaStream_t>(stream)));
}

int lazy_attn_pack_block_words_host(const lazy_attn_params* p, int32_t num_docs, const int32_t* seg_indptr,
                                    const int32_t* seg_doc, const int32_t* seg_len, const int32_t* seq_pos0,
                                    const int32_t* doc_block_indptr, const int32_t* doc_blocks,
                                    uint32_t* block_words, int32_t* seq_lens) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  const int B = p->num_seqs, MB = p->max_blocks_per_seq;
  if (num_docs < 0) return LAZY_ERR_INVALID_ARG;
  if (B > 0 && (!seg_indptr || !block_words || !seq_lens)) return LAZY_ERR_INVALID_ARG;
  if (B > 0 && seg_indptr[B] > seg_indptr[0] && (!seg_doc || !seg_len || !doc_block_indptr || !doc_blocks))
    return LAZY_ERR_INVALID_ARG;
  const uint32_t id_mask = (1u << c.id_bits) - 1u;
  const int64_t off_lo = -((int64_t)1 << (31 - c.id_bits)), off_hi = ((int64_t)1 << (31 - c.id_bits)) - 1;
  for (int s = 0; s < B; ++s) {
    uint32_t* wrow = block_words + (size_t)s * MB;
    const int k0 = seg_indptr[s], k1 = seg_indptr[s + 1];
    if (k1 < k0) return LAZY_ERR_LAYOUT;
    int64_t blk = 0, pos = seq_pos0 ? seq_pos0[s] : 0;
    int last_len = 0;
    for (int k = k0; k < k1; ++k) {
      const int doc = seg_doc[k], len = seg_len[k];
      if (doc < 0 || doc >= num_docs || len < 1) return LAZY_ERR_LAYOUT;
      const int dblk = doc_block_indptr[doc + 1] - doc_block_indptr[doc];
      if ((int64_t)len > (int64_t)lazy::kBlock * dblk) return LAZY_ERR_LAYOUT;
      const int nbk = (len + lazy::kBlock - 1) / lazy::kBlock;
      if (blk + nbk > MB) return LAZY_ERR_LAYOUT;
      for (int q = 0; q < nbk; ++q) {
        const int phys = doc_blocks[doc_block_indptr[doc] + q];
        // offset from the document's start, or (key_positions) from the block's first key
        const int64_t off = (int64_t)lazy::kBlock * (blk + q) - pos - (p->key_positions ? (int64_t)lazy::kBlock * q : 0);
        if (phys < 0 || phys >= p->num_pool_blocks || (uint32_t)phys > id_mask || off < off_lo || off > off_hi)
          return LAZY_ERR_LAYOUT;
        wrow[blk + q] = ((uint32_t)(int32_t)off << c.id_bits) | ((uint32_t)phys & id_mask);
      }
      blk += nbk;
      pos += len;
      last_len = len;
    }
    for (int64_t b = blk; b < MB; ++b) wrow[b] = 0u;
    const int last_blocks = (last_len + lazy::kBlock - 1) / lazy::kBlock;
    seq_lens[s] = blk == 0 ? 0 : (int32_t)(lazy::kBlock * blk - (lazy::kBlock * last_blocks - last_len));
  }
  return LAZY_OK;
}

int lazy_attn_pack_block_words(const lazy_attn_params* p, int32_t num_docs, const int32_t* seg_indptr,
                               const int32_t* seg_doc, const int32_t* seg_len, const int32_t* seq_pos0,
                               const int32_t* doc_block_indptr, const int32_t* doc_blocks, uint32_t* block_words,
                               int32_t* seq_lens, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (num_docs < 0) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return LAZY_OK;
  if (!seg_indptr || !seg_doc || !seg_len || !doc_block_indptr || !doc_blocks || !block_words || !seq_lens)
    return LAZY_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  lazy::PackArgs a{seg_indptr, seg_doc, seg_len, seq_pos0, doc_block_indptr, doc_blocks, block_words, seq_lens, st,
                   p->num_seqs, num_docs, p->max_blocks_per_seq, c.id_bits, p->num_pool_blocks, p->key_positions};
  return launched(lazy::launch_pack(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t lazy_attn_decode_workspace_bytes(const lazy_attn_params* p) {
  Checked c;
  if (check_params(p, &c) != LAZY_OK) return 0;
  int splits, bps;
  plan_splits(p, &splits, &bps);
  return decode_ws_bytes(p, splits);
}

static int decode_impl(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                       const uint32_t* block_words, const int32_t* seq_lens, const int32_t* q_pos,
                       const void* rope_table, const float* alibi, void* out, void* workspace,
                       size_t workspace_bytes, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  // key-position words carry no document start: only the ALiBi form reads them
  if (!alibi != !p->key_positions || (reinterpret_cast<uintptr_t>(alibi) & 3u)) return LAZY_ERR_INVALID_ARG;
  if (alibi && p->dtype != LAZY_BF16) return LAZY_ERR_UNSUPPORTED;
  const bool fp8 = kv_fp8(p);
  if (fp8 && (p->dtype != LAZY_BF16 || p->head_dim != 128 || alibi)) return LAZY_ERR_UNSUPPORTED;
  if (p->num_seqs == 0) return LAZY_OK;
  if (!q || !k_pool || !v_pool || !block_words || !seq_lens || !q_pos || !rope_table || !out)
    return LAZY_ERR_INVALID_ARG;
  if (p->num_pool_blocks == 0 || p->max_blocks_per_seq == 0) return LAZY_ERR_INVALID_ARG;
  if (p->dtype == LAZY_F32 && c.G > 32) return LAZY_ERR_UNSUPPORTED;
  if (p->dtype == LAZY_BF16 && c.G > 64) return LAZY_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) || !aligned16(rope_table))
    return LAZY_ERR_INVALID_ARG;
  int splits, bps;
  plan_splits(p, &splits, &bps);
  const size_t need = decode_ws_bytes(p, splits);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return LAZY_ERR_WORKSPACE;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  const size_t parts = (size_t)p->num_seqs * p->num_q_heads * splits;
  lazy::DecodeArgs a{};
  a.q = q;
  a.words = block_words;
  a.seq_lens = seq_lens;
  a.q_pos = q_pos;
  a.rope = static_cast<const float2*>(rope_table);
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.out = out;
  a.ws_o = need ? static_cast<float*>(workspace) : nullptr;
  a.ws_ml = need ? static_cast<float*>(workspace) + parts * p->head_dim : nullptr;
  a.status = st;
  a.B = p->num_seqs;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = c.G;
  a.D = p->head_dim;
  a.max_blocks = p->max_blocks_per_seq;
  a.id_bits = c.id_bits;
  a.num_pool_blocks = p->num_pool_blocks;
  a.splits = splits;
  a.bps = bps;
  a.scale_log2 = scale_log2(p);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (p->dtype == LAZY_F32) {
    rc = launched(lazy::launch_decode_f32(a, p->lazy != 0, cs));
  } else if (fp8) {
    CUtensorMap kmap, vmap;
    const uint64_t rows = (uint64_t)p->num_pool_blocks * p->num_kv_heads * lazy::kBlock;
    if (!encode_rows_map_fp8(&kmap, k_pool, rows, lazy::kBlock) || !encode_rows_map_fp8(&vmap, v_pool, rows, lazy::kBlock))
      return LAZY_ERR_CUDA;
    rc = launched(lazy::launch_decode_fp8(a, p->k_scale > 0.f ? p->k_scale : 1.f, p->v_scale > 0.f ? p->v_scale : 1.f,
                                          p->lazy != 0, kmap, vmap, cs));
  } else {
    CUtensorMap kmap, vmap;
    const uint64_t rows = (uint64_t)p->num_pool_blocks * p->num_kv_heads * lazy::kBlock;
    if (!encode_rows_map(&kmap, k_pool, rows, p->head_dim, lazy::kBlock) ||
        !encode_rows_map(&vmap, v_pool, rows, p->head_dim, lazy::kBlock))
      return LAZY_ERR_CUDA;
    rc = launched(lazy::launch_decode_bf16(a, alibi, p->lazy != 0, kmap, vmap, cs));
  }
  if (rc != LAZY_OK || splits == 1) return rc;
  return launched(lazy::launch_combine(a, p->dtype == LAZY_BF16, cs));
}

int lazy_attn_decode(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                     const uint32_t* block_words, const int32_t* seq_lens, const int32_t* q_pos,
                     const void* rope_table, void* out, void* workspace, size_t workspace_bytes,
                     lazy_stream_t stream) {
  return decode_impl(p, q, k_pool, v_pool, block_words, seq_lens, q_pos, rope_table, nullptr, out, workspace,
                     workspace_bytes, stream);
}

int lazy_attn_decode_alibi(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                           const uint32_t* block_words, const int32_t* seq_lens, const int32_t* q_pos,
                           const void* rope_table, const float* alibi_slopes, void* out, void* workspace,
                           size_t workspace_bytes, lazy_stream_t stream) {
  if (!alibi_slopes) return LAZY_ERR_INVALID_ARG;
  return decode_impl(p, q, k_pool, v_pool, block_words, seq_lens, q_pos, rope_table, alibi_slopes, out, workspace,
                     workspace_bytes, stream);
}

int lazy_attn_plan_shared_host(const lazy_attn_params* p, int32_t num_docs, const int32_t* seg_indptr,
                               const int32_t* seg_doc, const int32_t* seg_len, const int32_t* doc_block_indptr,
                               const int32_t* doc_blocks, int32_t chunk_blocks, int32_t capacity, int32_t* items,
                               int32_t* slot_indptr, int32_t* counts) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (num_docs < 0 || capacity < 0 || chunk_blocks < 0 || !slot_indptr || !counts) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs > 0 && !seg_indptr) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs > 0 && seg_indptr[p->num_seqs] > seg_indptr[0] &&
      (!seg_doc || !seg_len || !doc_block_indptr || !doc_blocks || !items))
    return LAZY_ERR_INVALID_ARG;
  if (c.G > 64) return LAZY_ERR_UNSUPPORTED;
  // e4m3 pools run on the mma.sync kernel (items of at most 64 rows) at every ratio
  const int cap = kv_fp8(p) ? 64 : lazy::shared_rows_cap(c.G, p->head_dim);
  // 0: 32 blocks for the mma.sync kernel; for the tensor-core kernel, a length that
  // gives about one item per resident CTA.
  const int cb = chunk_blocks > 0 ? chunk_blocks : (cap == 128 ? 0 : 32);
  const int auto_items = std::max(1, lazy::kSharedTcSlots / std::max(1, p->num_kv_heads));
  // small items spread through the launch: measured for the bf16 mma.sync kernel only
  const bool spread = !kv_fp8(p) && cap == 64;
  return lazy::plan_shared_host(p->num_seqs, c.G, cap, p->max_blocks_per_seq, p->num_pool_blocks, num_docs,
                                seg_indptr, seg_doc, seg_len, doc_block_indptr, doc_blocks, cb, auto_items, capacity,
                                items, slot_indptr, counts, spread);
}

size_t lazy_attn_decode_shared_workspace_bytes(const lazy_attn_params* p, int32_t num_slots) {
  Checked c;
  if (check_params(p, &c) != LAZY_OK || num_slots < 0) return 0;
  size_t bytes = (size_t)num_slots * p->num_q_heads * (p->head_dim + 2) * sizeof(float);
#ifdef LAZY_DECODE_TRACE
  bytes += (size_t)64 << 20;  // per-CTA trace counters
#endif
  return bytes;
}

// phase: kSharedBoth (work-item kernel, then the combine as its programmatic
// dependent), kSharedPartials (work-item kernel only), kSharedCombine (combine only).
enum { kSharedBoth = 0, kSharedPartials = 1, kSharedCombine = 2 };

static int decode_shared_impl(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                              const uint32_t* block_words, const int32_t* q_pos, const void* rope_table,
                              int32_t num_items, const int32_t* items, int32_t num_slots, const int32_t* slot_indptr,
                              const float* alibi, void* out, void* workspace, size_t workspace_bytes,
                              lazy_stream_t stream, int phase = kSharedBoth) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (!alibi != !p->key_positions || (reinterpret_cast<uintptr_t>(alibi) & 3u)) return LAZY_ERR_INVALID_ARG;
  if (p->dtype != LAZY_BF16) return LAZY_ERR_UNSUPPORTED;
  const bool fp8 = kv_fp8(p);
  if (fp8 && (p->head_dim != 128 || alibi)) return LAZY_ERR_UNSUPPORTED;
  if (c.G > 64) return LAZY_ERR_UNSUPPORTED;
  if (num_items < 0 || num_slots < 0) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return LAZY_OK;
  if (phase != kSharedCombine) {
    if (!q || !k_pool || !v_pool || !block_words || !q_pos || !rope_table) return LAZY_ERR_INVALID_ARG;
    if (num_items > 0 && (!items || num_slots == 0)) return LAZY_ERR_INVALID_ARG;
    if ((int64_t)num_items * p->num_kv_heads > INT32_MAX) return LAZY_ERR_UNSUPPORTED;
    if (p->num_pool_blocks == 0 || p->max_blocks_per_seq == 0) return LAZY_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(rope_table) ||
        (items && !aligned16(items)))
      return LAZY_ERR_INVALID_ARG;
  }
  if (phase != kSharedPartials && (!slot_indptr || !out || !aligned16(out))) return LAZY_ERR_INVALID_ARG;
  const size_t need = lazy_attn_decode_shared_workspace_bytes(p, num_slots);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return LAZY_ERR_WORKSPACE;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  lazy::SharedDecodeArgs a{};
  a.q = q;
  a.words = block_words;
  a.q_pos = q_pos;
  a.rope = static_cast<const float2*>(rope_table);
  a.items = items;
  a.slot_indptr = slot_indptr;
  a.out = out;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_ml = need ? static_cast<float*>(workspace) + (size_t)num_slots * p->num_q_heads * p->head_dim : nullptr;
  a.status = st;
  a.B = p->num_seqs;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = c.G;
  a.D = p->head_dim;
  a.max_blocks = p->max_blocks_per_seq;
  a.id_bits = c.id_bits;
  a.num_pool_blocks = p->num_pool_blocks;
  a.num_items = num_items;
  a.num_slots = num_slots;
  a.scale_log2 = scale_log2(p);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (phase == kSharedCombine) return launched(lazy::launch_shared_combine(a, cs));
  if (num_items > 0) {
    CUtensorMap kmap, vmap;
    const uint64_t rows = (uint64_t)p->num_pool_blocks * p->num_kv_heads * lazy::kBlock;
    if (fp8) {  // e4m3 codes: one 16-row x 128-byte box per block (mma.sync kernel at every ratio)
      if (!encode_rows_map_fp8(&kmap, k_pool, rows, lazy::kBlock) ||
          !encode_rows_map_fp8(&vmap, v_pool, rows, lazy::kBlock))
        return LAZY_ERR_CUDA;
      rc = launched(lazy::launch_decode_shared_fp8(a, p->k_scale > 0.f ? p->k_scale : 1.f,
                                                   p->v_scale > 0.f ? p->v_scale : 1.f, p->lazy != 0, kmap, vmap, cs));
    } else if (lazy::shared_rows_cap(c.G, p->head_dim) == 128) {  // tensor-core kernel: 16-row x 64-column boxes
      if (!encode_rows_map(&kmap, k_pool, rows, p->head_dim, lazy::kBlock) ||
          !encode_rows_map(&vmap, v_pool, rows, p->head_dim, lazy::kBlock))
        return LAZY_ERR_CUDA;
      rc = launched(lazy::launch_decode_shared_tc(a, alibi, alibi || p->lazy != 0, kmap, vmap, cs));
    } else {
      if (!encode_block_map(&kmap, k_pool, rows, p->head_dim, lazy::kBlock) ||
          !encode_block_map(&vmap, v_pool, rows, p->head_dim, lazy::kBlock))
        return LAZY_ERR_CUDA;
      rc = launched(lazy::launch_decode_shared(a, alibi, alibi || p->lazy != 0, kmap, vmap, cs));
    }
    if (rc != LAZY_OK) return rc;
  }
  if (phase == kSharedPartials) return LAZY_OK;
  return launched(lazy::launch_shared_combine(a, cs));
}

int lazy_attn_decode_shared_partials(const lazy_attn_params* p, const void* q, const void* k_pool,
                                     const void* v_pool, const uint32_t* block_words, const int32_t* q_pos,
                                     const void* rope_table, int32_t num_items, const int32_t* items,
                                     int32_t num_slots, void* workspace, size_t workspace_bytes,
                                     lazy_stream_t stream) {
  return decode_shared_impl(p, q, k_pool, v_pool, block_words, q_pos, rope_table, num_items, items, num_slots,
                            nullptr, nullptr, nullptr, workspace, workspace_bytes, stream, kSharedPartials);
}

int lazy_attn_decode_shared_combine(const lazy_attn_params* p, int32_t num_slots, const int32_t* slot_indptr,
                                    const void* workspace, size_t workspace_bytes, void* out, lazy_stream_t stream) {
  return decode_shared_impl(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, num_slots,
                            slot_indptr, nullptr, out, const_cast<void*>(workspace), workspace_bytes, stream,
                            kSharedCombine);
}

int lazy_attn_decode_shared(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                            const uint32_t* block_words, const int32_t* q_pos, const void* rope_table,
                            int32_t num_items, const int32_t* items, int32_t num_slots, const int32_t* slot_indptr,
                            void* out, void* workspace, size_t workspace_bytes, lazy_stream_t stream) {
  return decode_shared_impl(p, q, k_pool, v_pool, block_words, q_pos, rope_table, num_items, items, num_slots,
                            slot_indptr, nullptr, out, workspace, workspace_bytes, stream);
}

int lazy_attn_decode_shared_alibi(const lazy_attn_params* p, const void* q, const void* k_pool, const void* v_pool,
                                  const uint32_t* block_words, const int32_t* q_pos, const void* rope_table,
                                  int32_t num_items, const int32_t* items, int32_t num_slots,
                                  const int32_t* slot_indptr, const float* alibi_slopes, void* out, void* workspace,
                                  size_t workspace_bytes, lazy_stream_t stream) {
  if (!alibi_slopes) return LAZY_ERR_INVALID_ARG;
  return decode_shared_impl(p, q, k_pool, v_pool, block_words, q_pos, rope_table, num_items, items, num_slots,
                            slot_indptr, alibi_slopes, out, workspace, workspace_bytes, stream);
}

int lazy_attn_alibi_slopes_host(int32_t num_heads, float* out) {
  if (num_heads < 1 || num_heads > 4096 || !out) return LAZY_ERR_INVALID_ARG;
  // Geometric slopes 2^(-8 i / n), i = 1..n, for n a power of two; otherwise those of
  // the largest power of two n' below num_heads, then every other slope of 2 n'
  // (the odd-indexed ones) for the remaining heads.
  int np2 = 1;
  while (2 * np2 <= num_heads) np2 *= 2;
  for (int i = 0; i < np2; ++i) out[i] = (float)std::exp2(-8.0 * (double)(i + 1) / (double)np2);
  for (int k = 0; np2 + k < num_heads; ++k)
    out[np2 + k] = (float)std::exp2(-8.0 * (double)(2 * k + 1) / (double)(2 * np2));
  return LAZY_OK;
}

// The two-tile prefill (even GQA ratio) runs one persistent CTA per SM and needs a
// workspace for the pieces of units that cross CTA ranges; the one-tile kernel none.
static bool prefill_uses_stream(const lazy_attn_params* p, const Checked& c) {
  return p->dtype == LAZY_BF16 && p->head_dim == 128 && c.G % 2 == 0;
}

size_t lazy_attn_prefill_workspace_bytes(const lazy_attn_params* p, int32_t total_q) {
  (void)total_q;
  Checked c;
  if (check_params(p, &c) != LAZY_OK) return 0;
  if (!prefill_uses_stream(p, c)) return 0;
  return lazy::prefill_stream_workspace_bytes(current_device() >= 0 ? lazy::prefill_stream_grid() : kDefaultSmCount);
}

static int prefill_impl(const lazy_attn_params* p, const void* q, const int32_t* cu_seqlens_q, const int32_t* q_start,
                        int32_t total_q, int32_t max_q_len, const void* k_pool, const void* v_pool,
                        const uint32_t* block_words, const int32_t* seq_lens, const void* rope_table,
                        const float* alibi, void* out, void* workspace, size_t workspace_bytes, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (p->dtype != LAZY_BF16 || p->head_dim != 128 || kv_fp8(p)) return LAZY_ERR_UNSUPPORTED;
  // key-position words carry no document start: only the ALiBi form reads them
  if (total_q < 0 || max_q_len < 0 || !alibi != !p->key_positions || (reinterpret_cast<uintptr_t>(alibi) & 3u))
    return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs == 0 || total_q == 0 || max_q_len == 0) return LAZY_OK;
  if (!q || !cu_seqlens_q || !q_start || !k_pool || !v_pool || !block_words || !seq_lens || !rope_table || !out)
    return LAZY_ERR_INVALID_ARG;
  if (p->num_pool_blocks == 0 || p->max_blocks_per_seq == 0) return LAZY_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) || !aligned16(rope_table))
    return LAZY_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  CUtensorMap qmap, kmap, vmap;
  const uint64_t rows = (uint64_t)p->num_pool_blocks * p->num_kv_heads * lazy::kBlock;
  if (!encode_q_map(&qmap, q, (uint64_t)total_q, p->num_q_heads, p->head_dim, 128) ||
      !encode_rows_map(&kmap, k_pool, rows, p->head_dim, lazy::kBlock) ||
      !encode_rows_map(&vmap, v_pool, rows, p->head_dim, lazy::kBlock))
    return LAZY_ERR_CUDA;
  lazy::PrefillArgs a{};
  a.cu_seqlens_q = cu_seqlens_q;
  a.q_start = q_start;
  a.words = block_words;
  a.seq_lens = seq_lens;
  a.rope = static_cast<const float2*>(rope_table);
  a.out = out;
  a.status = st;
  a.B = p->num_seqs;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = c.G;
  a.D = p->head_dim;
  a.total_q = total_q;
  a.max_q_len = max_q_len;
  a.max_blocks = p->max_blocks_per_seq;
  a.id_bits = c.id_bits;
  a.num_pool_blocks = p->num_pool_blocks;
  a.scale_log2 = scale_log2(p);
  a.T = (max_q_len + lazy::pf_tile_rows - 1) / lazy::pf_tile_rows;
  int grid = 0;
  if (prefill_uses_stream(p, c)) {
    grid = lazy::prefill_stream_grid();
    const size_t need = lazy::prefill_stream_workspace_bytes(grid);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LAZY_ERR_WORKSPACE;
    a.counters = static_cast<int*>(workspace);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + lazy::prefill_stream_counter_bytes(grid));
  }
  cudaError_t e = lazy::launch_prefill(a, alibi ? false : p->lazy != 0, qmap, kmap, vmap, grid,
                                       reinterpret_cast<cudaStream_t>(stream), alibi);
  if (e == cudaErrorNotSupported) return LAZY_ERR_UNSUPPORTED;
  return launched(e);
}

int lazy_attn_prefill(const lazy_attn_params* p, const void* q, const int32_t* cu_seqlens_q, const int32_t* q_start,
                      int32_t total_q, int32_t max_q_len, const void* k_pool, const void* v_pool,
                      const uint32_t* block_words, const int32_t* seq_lens, const void* rope_table, void* out,
                      void* workspace, size_t workspace_bytes, lazy_stream_t stream) {
  return prefill_impl(p, q, cu_seqlens_q, q_start, total_q, max_q_len, k_pool, v_pool, block_words, seq_lens,
                      rope_table, nullptr, out, workspace, workspace_bytes, stream);
}

int lazy_attn_prefill_alibi(const lazy_attn_params* p, const void* q, const int32_t* cu_seqlens_q,
                            const int32_t* q_start, int32_t total_q, int32_t max_q_len, const void* k_pool,
                            const void* v_pool, const uint32_t* block_words, const int32_t* seq_lens,
                            const void* rope_table, const float* alibi_slopes, void* out, void* workspace,
                            size_t workspace_bytes, lazy_stream_t stream) {
  if (!alibi_slopes) return LAZY_ERR_INVALID_ARG;
  return prefill_impl(p, q, cu_seqlens_q, q_start, total_q, max_q_len, k_pool, v_pool, block_words, seq_lens,
                      rope_table, alibi_slopes, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- one launch for a mixed batch

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

static bool mixed_compatible(const lazy_attn_params* pd, const lazy_attn_params* pp, const Checked& cd) {
  return pd->num_q_heads == pp->num_q_heads && pd->num_kv_heads == pp->num_kv_heads &&
         pd->head_dim == pp->head_dim && pd->num_pool_blocks == pp->num_pool_blocks && pd->id_bits == pp->id_bits &&
         pd->dtype == pp->dtype && pd->sm_scale == pp->sm_scale && pd->lazy == pp->lazy &&
         pd->key_positions == pp->key_positions && pd->kv_dtype == pp->kv_dtype && pd->head_dim == 128 &&
         pd->dtype == LAZY_BF16 && !kv_fp8(pd) && pd->lazy != 0 && !pd->key_positions && cd.G % 16 == 0 &&
         lazy::shared_rows_cap(cd.G, pd->head_dim) == 128;
}

size_t lazy_attn_mixed_workspace_bytes(const lazy_attn_params* p_dec, const lazy_attn_params* p_pf, int32_t num_slots) {
  Checked cd, cp;
  if (check_params(p_dec, &cd) != LAZY_OK || check_params(p_pf, &cp) != LAZY_OK || num_slots < 0) return 0;
  const int grid = current_device() >= 0 ? lazy::prefill_stream_grid() : kDefaultSmCount;
  return align256(lazy::prefill_stream_workspace_bytes(grid)) +
         align256((size_t)num_slots * p_dec->num_q_heads * (p_dec->head_dim + 2) * sizeof(float)) +
         align256((size_t)p_dec->num_seqs * sizeof(int));
}

int lazy_attn_mixed(const lazy_attn_params* p_dec, const void* q_dec, const uint32_t* words_dec, const int32_t* q_pos,
                    int32_t num_items, const int32_t* items, int32_t num_slots, const int32_t* slot_indptr,
                    void* out_dec, const lazy_attn_params* p_pf, const void* q_pf, const int32_t* cu_seqlens_q,
                    const int32_t* q_start, int32_t total_q, int32_t max_q_len, const uint32_t* words_pf,
                    const int32_t* seq_lens_pf, void* out_pf, const void* k_pool, const void* v_pool,
                    const void* rope_table, void* workspace, size_t workspace_bytes, lazy_stream_t stream) {
  Checked cd, cp;
  int rc = check_params(p_dec, &cd);
  if (rc != LAZY_OK) return rc;
  rc = check_params(p_pf, &cp);
  if (rc != LAZY_OK) return rc;
  if (!mixed_compatible(p_dec, p_pf, cd)) return LAZY_ERR_UNSUPPORTED;
  if (num_items < 0 || num_slots < 0 || total_q < 0 || max_q_len < 0) return LAZY_ERR_INVALID_ARG;
  // A batch with only one kind of work is the plain call of that kind.
  if (p_pf->num_seqs == 0 || total_q == 0 || max_q_len == 0)
    return lazy_attn_decode_shared(p_dec, q_dec, k_pool, v_pool, words_dec, q_pos, rope_table, num_items, items,
                                   num_slots, slot_indptr, out_dec, workspace, workspace_bytes, stream);
  if (p_dec->num_seqs == 0) {
    const size_t need = lazy_attn_prefill_workspace_bytes(p_pf, total_q);
    return lazy_attn_prefill(p_pf, q_pf, cu_seqlens_q, q_start, total_q, max_q_len, k_pool, v_pool, words_pf,
                             seq_lens_pf, rope_table, out_pf, workspace, workspace_bytes < need ? 0 : workspace_bytes,
                             stream);
  }
  if (!q_dec || !words_dec || !q_pos || !slot_indptr || !out_dec || !q_pf || !cu_seqlens_q || !q_start || !words_pf ||
      !seq_lens_pf || !out_pf || !k_pool || !v_pool || !rope_table)
    return LAZY_ERR_INVALID_ARG;
  if (num_items > 0 && (!items || num_slots == 0)) return LAZY_ERR_INVALID_ARG;
  if ((int64_t)num_items * p_dec->num_kv_heads > INT32_MAX) return LAZY_ERR_UNSUPPORTED;
  if (p_dec->num_pool_blocks == 0 || p_dec->max_blocks_per_seq == 0 || p_pf->max_blocks_per_seq == 0)
    return LAZY_ERR_INVALID_ARG;
  if (!aligned16(q_dec) || !aligned16(q_pf) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out_dec) ||
      !aligned16(out_pf) || !aligned16(rope_table) || (items && !aligned16(items)))
    return LAZY_ERR_INVALID_ARG;
  const int grid = lazy::prefill_stream_grid();
  const size_t pf_bytes = align256(lazy::prefill_stream_workspace_bytes(grid));
  const size_t dec_bytes = align256((size_t)num_slots * p_dec->num_q_heads * (p_dec->head_dim + 2) * sizeof(float));
  const size_t need = lazy_attn_mixed_workspace_bytes(p_dec, p_pf, num_slots);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return LAZY_ERR_WORKSPACE;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  CUtensorMap qmap, qmap_dec, kmap, vmap;
  const uint64_t rows = (uint64_t)p_pf->num_pool_blocks * p_pf->num_kv_heads * lazy::kBlock;
  // decode queries [B_dec][Hq][d]: one box is the G query heads of one KV head of one sequence
  if (!encode_q_map(&qmap, q_pf, (uint64_t)total_q, p_pf->num_q_heads, p_pf->head_dim, 128) ||
      !encode_dec_q_map(&qmap_dec, q_dec, (uint64_t)p_dec->num_seqs, p_dec->num_q_heads, p_dec->head_dim, cd.G) ||
      !encode_rows_map(&kmap, k_pool, rows, p_pf->head_dim, lazy::kBlock) ||
      !encode_rows_map(&vmap, v_pool, rows, p_pf->head_dim, lazy::kBlock))
    return LAZY_ERR_CUDA;
  lazy::MixedArgs a{};
  a.cu_seqlens_q = cu_seqlens_q;
  a.q_start = q_start;
  a.words = words_pf;
  a.seq_lens = seq_lens_pf;
  a.rope = static_cast<const float2*>(rope_table);
  a.out = out_pf;
  a.status = st;
  a.B = p_pf->num_seqs;
  a.Hq = p_pf->num_q_heads;
  a.Hkv = p_pf->num_kv_heads;
  a.G = cp.G;
  a.D = p_pf->head_dim;
  a.total_q = total_q;
  a.max_q_len = max_q_len;
  a.max_blocks = p_pf->max_blocks_per_seq;
  a.id_bits = cp.id_bits;
  a.num_pool_blocks = p_pf->num_pool_blocks;
  a.scale_log2 = scale_log2(p_pf);
  a.T = (max_q_len + lazy::pf_tile_rows - 1) / lazy::pf_tile_rows;
  a.counters = static_cast<int*>(workspace);
  a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + lazy::prefill_stream_counter_bytes(grid));
  a.q_dec = q_dec;
  a.words_dec = words_dec;
  a.q_pos = q_pos;
  a.items = items;
  a.slot_indptr = slot_indptr;
  a.out_dec = out_dec;
  a.ws_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + pf_bytes);
  a.ws_ml = a.ws_o + (size_t)num_slots * p_dec->num_q_heads * p_dec->head_dim;
  a.seq_done = reinterpret_cast<int*>(static_cast<char*>(workspace) + pf_bytes + dec_bytes);
  a.B_dec = p_dec->num_seqs;
  a.max_blocks_dec = p_dec->max_blocks_per_seq;
  a.num_items = num_items;
  a.num_slots = num_slots;
  cudaError_t e = lazy::launch_mixed(a, qmap, qmap_dec, kmap, vmap, grid, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return LAZY_ERR_UNSUPPORTED;
  return launched(e);
}

int lazy_attn_materialize(const lazy_attn_params* p, const void* k_pool, const void* v_pool,
                          const uint32_t* block_words, const int32_t* seq_lens, const void* rope_table, void* k_out,
                          void* v_out, uint32_t* block_words_out, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (p->dtype != LAZY_BF16 || kv_fp8(p)) return LAZY_ERR_UNSUPPORTED;
  if (p->key_positions) return LAZY_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return LAZY_OK;
  if (!k_pool || !v_pool || !block_words || !seq_lens || !rope_table || !k_out || !v_out || !block_words_out)
    return LAZY_ERR_INVALID_ARG;
  if (p->num_pool_blocks == 0 || p->max_blocks_per_seq == 0) return LAZY_ERR_INVALID_ARG;
  if ((int64_t)p->num_seqs * p->max_blocks_per_seq > ((int64_t)1 << c.id_bits)) return LAZY_ERR_LAYOUT;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_out) || !aligned16(v_out) || !aligned16(rope_table))
    return LAZY_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  lazy::MaterializeArgs a{k_pool, v_pool, block_words, seq_lens, static_cast<const float2*>(rope_table), k_out, v_out,
                          block_words_out, st, p->num_seqs, p->num_kv_heads, p->head_dim, p->max_blocks_per_seq,
                          c.id_bits, p->num_pool_blocks};
  return launched(lazy::launch_materialize(a, reinterpret_cast<cudaStream_t>(stream)));
}

static int debug_gather_impl(const lazy_attn_params* p, const void* k_pool, const void* v_pool,
                             const uint32_t* block_words, const int32_t* seq_lens, void* k_out, void* v_out,
                             int32_t* pos_out, int32_t withhold_block, uint64_t wait_ns, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (kv_fp8(p)) return LAZY_ERR_UNSUPPORTED;
  if (p->num_seqs == 0) return LAZY_OK;
  if (!k_pool || !v_pool || !block_words || !seq_lens || !k_out || !v_out) return LAZY_ERR_INVALID_ARG;
  if (p->num_pool_blocks == 0 || p->max_blocks_per_seq == 0) return LAZY_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_out) || !aligned16(v_out)) return LAZY_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  lazy::GatherArgs a{block_words, seq_lens, k_pool, v_pool, k_out, v_out, pos_out, st,
                     p->num_seqs, p->num_kv_heads, p->head_dim, p->max_blocks_per_seq, c.id_bits,
                     p->num_pool_blocks, withhold_block, wait_ns};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (p->dtype == LAZY_F32) {
    if (withhold_block >= 0) return LAZY_ERR_UNSUPPORTED;  // the fp32 gather has no pipeline to stall
    return launched(lazy::launch_gather_f32(a, cs));
  }
  CUtensorMap kmap, vmap;
  const uint64_t rows = (uint64_t)p->num_pool_blocks * p->num_kv_heads * lazy::kBlock;
  if (!encode_rows_map(&kmap, k_pool, rows, p->head_dim, lazy::kBlock) ||
      !encode_rows_map(&vmap, v_pool, rows, p->head_dim, lazy::kBlock))
    return LAZY_ERR_CUDA;
  return launched(lazy::launch_gather_bf16(a, kmap, vmap, cs));
}

int lazy_attn_debug_gather(const lazy_attn_params* p, const void* k_pool, const void* v_pool,
                           const uint32_t* block_words, const int32_t* seq_lens, void* k_out, void* v_out,
                           int32_t* pos_out, lazy_stream_t stream) {
  return debug_gather_impl(p, k_pool, v_pool, block_words, seq_lens, k_out, v_out, pos_out, -1, lazy::kWaitLimitNs,
                           stream);
}

int lazy_attn_debug_gather_withheld(const lazy_attn_params* p, const void* k_pool, const void* v_pool,
                                    const uint32_t* block_words, const int32_t* seq_lens, void* k_out, void* v_out,
                                    int32_t* pos_out, int32_t withhold_block, uint32_t wait_limit_us,
                                    lazy_stream_t stream) {
  if (withhold_block < 0 || wait_limit_us == 0 || (uint64_t)wait_limit_us * 1000u > lazy::kWaitLimitNs)
    return LAZY_ERR_INVALID_ARG;
  return debug_gather_impl(p, k_pool, v_pool, block_words, seq_lens, k_out, v_out, pos_out, withhold_block,
                           (uint64_t)wait_limit_us * 1000u, stream);
}

int lazy_attn_debug_rope(const lazy_attn_params* p, const void* rope_table, const int32_t* deltas, int32_t n,
                         void* cs_out, lazy_stream_t stream) {
  Checked c;
  int rc = check_params(p, &c);
  if (rc != LAZY_OK) return rc;
  if (n < 0) return LAZY_ERR_INVALID_ARG;
  if (n == 0) return LAZY_OK;
  if (!rope_table || !deltas || !cs_out || !aligned16(rope_table)) return LAZY_ERR_INVALID_ARG;
  unsigned int* st = status_ptr();
  if (!st) return LAZY_ERR_CUDA;
  return launched(lazy::launch_debug_rope(static_cast<const float2*>(rope_table), deltas, n, p->head_dim,
                                          static_cast<float2*>(cs_out), st, reinterpret_cast<cudaStream_t>(stream)));
}

int lazy_attn_device_status(uint32_t* flags_out, int clear) {
  if (!flags_out) return LAZY_ERR_INVALID_ARG;
  if (!status_ptr()) return LAZY_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return LAZY_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_lazy_status, sizeof v) != cudaSuccess) return LAZY_ERR_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_lazy_status, &zero, sizeof zero) != cudaSuccess) return LAZY_ERR_CUDA;
  }
  *flags_out = v;
  return LAZY_OK;
}

}  // extern "C"
