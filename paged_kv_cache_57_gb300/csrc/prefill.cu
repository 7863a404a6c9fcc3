// prefill.cu -- LazyAttention prefill on the 5th-generation tensor cores (sm_103a):
// choice of kernel.
//
// Technical summary "Resumo Técnico: LazyAttention", "Implementação Técnica",
// item 1 (Prefilling, compute-bound): K blocks are loaded from the
// position-agnostic cache and each receives ONE relative rotation (by R_p of its
// document, since stored K already carries its local position) instead of an
// unrotate-then-rerotate pass; the query tile is rotated once by R_m. The extra
// work is 3*N*d FLOPs per N-key tile against 4*M*N*d for the tile's two matrix
// products, i.e. 3/(4M): 0.59% at M = 128 rows per rotated key tile.
//
// Two kernels compute it:
//   prefill_stream.cu  two query tiles per CTA (q-heads h, h+1 of one KV head), so
//                      each loaded and rotated K/V tile serves 256 query rows; one
//                      persistent CTA per SM over a stream-K split of the work;
//                      needs an even GQA ratio.
//   prefill_tq.cu      one query tile per CTA with Q' held in tensor memory; any
//                      GQA ratio.
// With ALiBi ("Principais Contribuições", item 4: the mechanism carries over to
// relative encodings such as ALiBi) both run without rotation on key-position block
// words, and the softmax adds slope_h (n - m) to each score from the block's first
// key position and the slot.
#include "kernels.h"

namespace lazy {

cudaError_t launch_prefill(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int grid, cudaStream_t st, const float* alibi) {
  if (a.D != 128) return cudaErrorNotSupported;
  if (alibi && lazy) return cudaErrorInvalidValue;  // ALiBi: key-position words, no rotation
  if (a.B == 0 || a.max_q_len == 0) return cudaSuccess;
  if (a.G % 2 == 0) return launch_prefill_stream(a, lazy, qmap, kmap, vmap, grid, st, alibi);
  return launch_prefill_tq(a, lazy, qmap, kmap, vmap, st, alibi);
}

}  // namespace lazy
