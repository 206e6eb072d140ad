// tc_linear.cu -- tensor-core path (filled in by the tcgen05 kernels).
#include "common.cuh"
#include "tc.cuh"

namespace poetx {

bool tc_cnp_supported(int, poetx_dtype) { return false; }
poetx_status tc_cnp_fwd(const float*, int, int, int, void*, poetx_dtype, cudaStream_t) {
  return POETX_ERR_UNSUPPORTED;
}
bool tc_linear_supported(int, int, int, int, poetx_dtype) { return false; }
size_t tc_workspace_bytes(int, int, int, int, int, poetx_dtype, bool) { return 0; }
poetx_status tc_forward(const void*, const void*, const void*, const void*, const int32_t*,
                        const int32_t*, const int32_t*, const int32_t*, int, int, int, int, int,
                        void*, void*, void*, void*, cudaStream_t) {
  return POETX_ERR_UNSUPPORTED;
}
poetx_status tc_backward(const void*, const void*, const void*, const void*, const void*,
                         const void*, const int32_t*, const int32_t*, const int32_t*,
                         const int32_t*, int, int, int, int, int, void*, void*, void*, float*,
                         float*, void*, cudaStream_t) {
  return POETX_ERR_UNSUPPORTED;
}

}  // namespace poetx
