// prefill.cu -- LazyAttention prefill (tcgen05 / TMEM, sm_103a).
#include "common.cuh"
#include "kernels.h"

namespace lazy {

cudaError_t launch_prefill(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t st) {
  (void)a, (void)lazy, (void)qmap, (void)kmap, (void)vmap, (void)st;
  return cudaErrorNotSupported;
}

}  // namespace lazy
