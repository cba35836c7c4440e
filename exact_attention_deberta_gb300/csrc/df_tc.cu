// Tensor-core (tcgen05 / TMEM / TMA) fused forward for bf16 and fp16.
#include "df_common.cuh"

namespace dfa {

bool tc_enabled() { return false; }

cudaError_t launch_tc(const Problem&, cudaStream_t, cudaEvent_t, cudaEvent_t, int* launches) {
  *launches = 0;
  return cudaErrorNotSupported;
}

}  // namespace dfa
