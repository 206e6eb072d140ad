// quant.cu -- POET-XQ: the frozen weight kept in INT8, dequantised per use.
//
// [POET-X §2.E] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, section 2.E): the base
// weight can be stored in INT8 and dequantised on the fly.  The page gives no
// scale granularity; here every row of the (merged) weight has one fp32 scale,
// symmetric, codes in [-127, 127]:
//   s_i = max_k |W[i][k]| / 127          (fp32, correctly rounded division)
//   q[i][k] = rint(W[i][k] / s_i)        (fp32 division, round half to even;
//                                         a row of zeros has s_i = 0, q = 0)
//   W'[i][k] = q[i][k] * s_i             (fp32 product, rounded to the
//                                         activation dtype)
// A row permutation or a column permutation of W permutes the codes and the
// scales the same way, so quantising the merged weight equals merging the
// quantised weight.  Dequantisation writes the activation-dtype weight into a
// scratch region right before the products that read it: at 1 + 2 bytes per
// element it is a short HBM-bound pass whose output is still in L2 when the
// tensor-core GEMM loads it, whereas converting inside the GEMM's load path
// would put a second read and write of every B tile on the shared memory
// that feeds the tensor core.
#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace poetx {

namespace {

constexpr int kQuantThreads = 256;

template <typename T>
__device__ __forceinline__ float load_f(const T* p) {
  return static_cast<float>(*p);
}
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// One CTA per row: the row's absolute maximum, its scale, then its codes.
template <typename T>
__global__ void __launch_bounds__(kQuantThreads) quantize_rows_kernel(const T* __restrict__ W,
                                                                      int d_in, int8_t* __restrict__ q,
                                                                      float* __restrict__ scale) {
  __shared__ float warp_max[kQuantThreads / 32];
  const int i = blockIdx.x;
  const T* row = W + (size_t)i * d_in;
  float m = 0.f;
  for (int k = threadIdx.x; k < d_in; k += kQuantThreads) m = fmaxf(m, fabsf(load_f(row + k)));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x / 32] = m;
  __syncthreads();
  m = warp_max[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
  const float s = __fdiv_rn(m, 127.f);
  if (threadIdx.x == 0) scale[i] = s;
  int8_t* qrow = q + (size_t)i * d_in;
  for (int k = threadIdx.x; k < d_in; k += kQuantThreads) {
    int c = 0;
    if (s > 0.f) {
      c = __float2int_rn(__fdiv_rn(load_f(row + k), s));
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
    }
    qrow[k] = (int8_t)c;
  }
}

__device__ __forceinline__ void store_deq(float* dst, const float* v) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store_deq(__nv_bfloat16* dst, const float* v) {
  __nv_bfloat162 h[2] = {__floats2bfloat162_rn(v[0], v[1]), __floats2bfloat162_rn(v[2], v[3])};
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
}

// W'[i][k] = q[i][k] * s_i, V codes per thread (V = 16 when d_in % 16 == 0:
// one 16-byte load of codes and two (bf16) or four (fp32) 16-byte stores;
// else V = 4); grid-stride over the matrix.
template <typename T, int V>
__global__ void __launch_bounds__(kQuantThreads) dequantize_kernel(const int8_t* __restrict__ q,
                                                                   const float* __restrict__ scale,
                                                                   int d_out, int d_in,
                                                                   T* __restrict__ W) {
  const size_t groups = (size_t)d_out * d_in / V;
  const int row_groups = d_in / V;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < groups;
       e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / row_groups);
    const float s = __ldg(scale + i);
    uint32_t c[V / 4];
    if constexpr (V == 16) {
      const uint4 c16 = __ldg(reinterpret_cast<const uint4*>(q) + e);
      c[0] = c16.x; c[1] = c16.y; c[2] = c16.z; c[3] = c16.w;
    } else {
      c[0] = __ldg(reinterpret_cast<const uint32_t*>(q) + e);
    }
#pragma unroll
    for (int w = 0; w < V / 4; ++w) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fmul_rn((float)(int8_t)(c[w] >> (8 * j)), s);
      store_deq(W + e * V + w * 4, v);
    }
  }
}

}  // namespace

poetx_status launch_quantize_w0(const void* W, int d_out, int d_in, poetx_dtype dt, int8_t* q,
                                float* scale, cudaStream_t s) {
  if (d_out <= 0 || d_in <= 0) return POETX_OK;
  {
    KernelScope ks_("quantize_w0", s);
    if (dt == POETX_F32)
      quantize_rows_kernel<float><<<d_out, kQuantThreads, 0, s>>>((const float*)W, d_in, q, scale);
    else
      quantize_rows_kernel<__nv_bfloat16><<<d_out, kQuantThreads, 0, s>>>(
          (const __nv_bfloat16*)W, d_in, q, scale);
  }
  return check_launch();
}

poetx_status launch_dequantize_w0(const int8_t* q, const float* scale, int d_out, int d_in,
                                  poetx_dtype dt, void* W, cudaStream_t s) {
  if (d_out <= 0 || d_in <= 0) return POETX_OK;
  if (d_in % 4) return POETX_ERR_SHAPE;
  const bool v16 = d_in % 16 == 0;
  const size_t groups = (size_t)d_out * d_in / (v16 ? 16 : 4);
  // one group per thread while that fills every SM several times over
  size_t blocks = (groups + kQuantThreads - 1) / kQuantThreads;
  const size_t cap = (size_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const unsigned nb = (unsigned)blocks;
  {
    KernelScope ks_("dequantize_w0", s);
    if (dt == POETX_F32) {
      if (v16) dequantize_kernel<float, 16><<<nb, kQuantThreads, 0, s>>>(q, scale, d_out, d_in, (float*)W);
      else dequantize_kernel<float, 4><<<nb, kQuantThreads, 0, s>>>(q, scale, d_out, d_in, (float*)W);
    } else {
      __nv_bfloat16* Wb = (__nv_bfloat16*)W;
      if (v16) dequantize_kernel<__nv_bfloat16, 16><<<nb, kQuantThreads, 0, s>>>(q, scale, d_out, d_in, Wb);
      else dequantize_kernel<__nv_bfloat16, 4><<<nb, kQuantThreads, 0, s>>>(q, scale, d_out, d_in, Wb);
    }
  }
  return check_launch();
}

}  // namespace poetx
