// Placeholder definitions until the tensor-core kernels land (shapes report unsupported).
#include "hyb_internal.cuh"
namespace hyb {
bool linear_prefill_tc_supported(int, int, int) { return false; }
cudaError_t launch_linear_prefill_tc(void*, const void*, const void*, const void*, const int32_t*,
                                     const int32_t*, float*, int, const int32_t*, const uint8_t*,
                                     int, int, int, int, int, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}
bool prefill_tc_supported(int, int) { return false; }
cudaError_t launch_prefill_tc(void*, const void*, const void*, const void*, const int32_t*,
                              const int32_t*, const int32_t*, int, int, int, int, int, int, float,
                              unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace hyb
