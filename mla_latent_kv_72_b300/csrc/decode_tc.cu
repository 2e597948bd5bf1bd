// mla_decode_fwd, tensor-core kernel (tcgen05 / TMEM / TMA) - not built yet.
#include "common.cuh"

namespace mla {

bool decode_tc_supported(int, const mla_kv_cache&, int) { return false; }

cudaError_t launch_decode_tc(const void*, const mla_kv_cache&, const int32_t*, int,
                             const int32_t*, int, int, int, float, float*, float*, int32_t*,
                             cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
