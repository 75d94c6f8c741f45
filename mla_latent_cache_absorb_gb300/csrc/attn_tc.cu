// tcgen05 split attention (bf16 rows, tensor cores). Not built yet: the CUDA-core path runs.
#include "common.cuh"

namespace mla {

bool attn_tc_supported(const mla_config& cfg) {
  (void)cfg;
  return false;
}

cudaError_t launch_attn_tc(const mla_config&, const mla_cache&, const DecodePlan&, const int32_t*,
                           const void*, float*, float*, int, WsHeader*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
