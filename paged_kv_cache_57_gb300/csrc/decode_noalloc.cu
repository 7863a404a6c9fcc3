// decode_noalloc.cu -- decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a serving engine that
// has reserved nearly all of HBM for its KV-cache pool and keeps no spare
// allocation, a plugin running inside another framework that may only use that
// framework's buffers, or a latency-critical step that must not call cudaMalloc
// (it can synchronise the device). For them this file provides a decode entry
// point whose split-K scratch is a file-scope static device array, created with
// the library and held by every GPU that loads it until the process exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/lazy_attn.h"

namespace {

// Split partials of one call: [B][Hq][splits][d] running outputs, then
// [B][Hq][splits][2] (max, sum). Every element the combine pass reads is written
// earlier in the same call, so nothing needs clearing between calls.
__device__ __align__(256) unsigned char g_decode_scratch[LAZY_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchEntry {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none yet)
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

bool driver_calls_ready() {  // under g_mu
  if (g_ctx_current && g_ctx_id) return true;
  void* a = nullptr;
  void* b = nullptr;
  cudaDriverEntryPointQueryResult qa, qb;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
      qa != cudaDriverEntryPointSuccess || !a ||
      cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
      qb != cudaDriverEntryPointSuccess || !b)
    return false;
  g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
  g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
  return true;
}

// Device address of the scratch array in the current device's context. In host
// code the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, with the device current. The lookup is cached per
// device together with the unique id of the context it was made in, and redone
// when that context has changed (after cudaDeviceReset, or when a caller made
// another context current): an address from an earlier context would point at
// memory that no longer holds the array.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!driver_calls_ready()) return nullptr;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return nullptr;
  if (!ctx) {  // no context current yet: the runtime creates the device's own on its next call
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
  }
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS || id == 0) return nullptr;
  ScratchEntry& e = g_scratch[dev];
  if (e.ctx_id != id || !e.ptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
    e = ScratchEntry{id, ptr};
  }
  return e.ptr;
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
