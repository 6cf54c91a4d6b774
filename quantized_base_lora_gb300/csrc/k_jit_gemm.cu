// K3: prefill GEMM of the per-layer JIT path (placeholder until the tcgen05
// kernel lands; the JIT path reports "not supported").
#include "ovl_internal.h"

namespace ovl {

size_t jit_gemm_x_scratch_bytes(uint32_t T, uint32_t n) { return size_t(T) * n * 4; }

cudaError_t launch_jit_gemm(const float*, const void*, uint32_t, uint32_t, uint32_t, uint32_t, float*,
                            float*, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ovl
