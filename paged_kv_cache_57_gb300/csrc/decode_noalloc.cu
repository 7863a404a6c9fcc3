// decode_noalloc.cu -- decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a serving engine that
// has reserved nearly all of HBM for its KV-cache pool and keeps no spare
// allocation, a plugin running inside another framework that may only use that
// framework's buffers, or a latency-critical step that must not call cudaMalloc
// (it can synchronise the device). For them this file provides a decode entry
// point whose split-K scratch is a file-scope static device array, created with
// the library and held by every GPU that loads it until the process exits.
#include <mutex>

#include "../../include/lazy_attn.h"

namespace {

// Split partials of one call: [B][Hq][splits][d] running outputs, then
// [B][Hq][splits][2] (max, sum). Every element the combine pass reads is written
// earlier in the same call, so nothing needs clearing between calls.
__device__ __align__(256) unsigned char g_decode_scratch[LAZY_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int lazy_attn_decode_noalloc(const lazy_attn_params* p, const void* q, const void* k_pool,
                                        const void* v_pool, const uint32_t* block_words, const int32_t* seq_lens,
                                        const int32_t* q_pos, const void* rope_table, void* out,
                                        lazy_stream_t stream) {
  if (!p) return LAZY_ERR_INVALID_ARG;
  const size_t need = lazy_attn_decode_workspace_bytes(p);
  if (need > (size_t)LAZY_NOALLOC_SCRATCH_BYTES) return LAZY_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_address();
    if (!scratch) return LAZY_ERR_CUDA;
  }
  return lazy_attn_decode(p, q, k_pool, v_pool, block_words, seq_lens, q_pos, rope_table, out, scratch,
                          need > 0 ? (size_t)LAZY_NOALLOC_SCRATCH_BYTES : 0, stream);
}
