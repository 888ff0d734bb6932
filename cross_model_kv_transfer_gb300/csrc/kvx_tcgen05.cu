// kvx_tcgen05.cu -- tensor-core (tcgen05) transfer kernel for bf16 caches.
#include <cuda_runtime.h>

#include "kvx_internal.h"

bool kvx_tc_supports(const kvx_plan_desc &) { return false; }
cudaError_t kvx_tc_prepare(const kvx_plan *) { return cudaErrorNotSupported; }
cudaError_t kvx_tc_launch(const kvx_plan *, const KvxParams &, cudaStream_t) {
  return cudaErrorNotSupported;
}
