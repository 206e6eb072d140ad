// common.cuh -- shared device helpers of the POET-X B300 library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "poetx.h"

namespace poetx {

// ---------------------------------------------------------------- element access
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Packed index of the strict-upper-triangle entry (i, k), i < k, of a b x b
// block: rows are stored one after another, row i holding b-1-i entries.
__device__ __forceinline__ int skew_index(int i, int k, int b) {
  return i * b - ((i * (i + 1)) >> 1) + (k - i - 1);
}

// K[r][c] of one block from its packed parameters (row-major upper triangle).
__device__ __forceinline__ float skew_entry(const float* __restrict__ theta, int r, int c, int b) {
  if (r < c) return __ldg(theta + skew_index(r, c, b));
  if (r > c) return -__ldg(theta + skew_index(c, r, b));
  return 0.0f;
}

// ---------------------------------------------------------------- device error word
// Kernels whose waits are bounded receive the address of the library's device
// error word; on an expired wait they record POETX_ERR_TIMEOUT there (first
// error wins).  poetx_stream_status() reads and clears it.
__device__ __forceinline__ void raise_device_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace poetx

// ---------------------------------------------------------------- host helpers
namespace poetx {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
inline size_t dtype_size(poetx_dtype d) { return d == POETX_F32 ? 4 : 2; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Records the last CUDA error of this library's launches; returns POETX_ERR_CUDA on error.
poetx_status check_launch();

// Device address of the error word on the current device (nullptr on failure).
int* device_error_word();

// Launch set-up that does not change between calls, done once (launch.cu):
// the multiprocessor count of the current device; the dynamic shared memory
// limit of a kernel (set once per device, kernel and size); the number of
// clusters of a kernel's launch configuration that fit on the device at once
// (0 if none or on error).
int device_sm_count();
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);
int max_active_clusters(const void* kernel, const cudaLaunchConfig_t& cfg);

}  // namespace poetx
