// cnp_simt.cu -- Cayley-Neumann parameterisation on the CUDA cores (fp32 FFMA).
//
// [POET-X §2.D] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.D): each b x b block is
// Q = (I + K)(I + K + ... + K^n) with K skew-symmetric, stored as the b(b-1)/2
// entries of its strict upper triangle.  The page fuses the Neumann chain into
// one kernel that keeps K and its powers on chip; here one CTA owns a slab of
// rows of one block and carries its rows of K^m from power to power in shared
// memory, streaming K itself through shared memory in row chunks unpacked
// straight from the packed parameters (the dense K never touches HBM).
//
// This is the exact-fp32 path (any power-of-two b <= 256).  The forward
// serves the block sizes the tensor-core kernels do not take: b <= 16, fp32 Q
// at b = 256, and bf16 Q at b = 256 beyond 65535 blocks; the backward serves
// the standalone poetx_cayley_neumann_backward and the fp32 layer.
#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace poetx {

namespace {

constexpr int kThreads = 256;
constexpr int kRowSlab = 16;   // rows of Q per CTA (forward)
constexpr int kColSlab = 16;   // columns of dK per CTA (backward)
constexpr int kChunk = 32;     // rows of K staged per step

// Stage rows [k0, k0 + kc) of K (all b columns) into shared memory.
//   transposed == false: dst[kk * ld + c] = K[k0 + kk][c]
//   transposed == true : dst[c * ld + kk] = K[k0 + kk][c]
// Entries above the diagonal (c > k) come from packed row k (contiguous in c);
// entries below (c < k) are -theta(c, k), read along packed row c, which is
// contiguous in k, so both halves are read with unit stride.
__device__ void stage_skew_rows(const float* __restrict__ theta, int b, int k0, int kc,
                                float* dst, int ld, bool transposed) {
  // upper part, c > k: packed row k, consecutive threads take consecutive c
  for (int e = threadIdx.x; e < kc * b; e += blockDim.x) {
    const int kk = e / b, c = e % b, k = k0 + kk;
    if (c > k) {
      const float v = __ldg(theta + skew_index(k, c, b));
      if (transposed) dst[c * ld + kk] = v; else dst[kk * ld + c] = v;
    } else if (c == k) {
      if (transposed) dst[c * ld + kk] = 0.f; else dst[kk * ld + c] = 0.f;
    }
  }
  // lower part, c < k: packed row c, consecutive threads take consecutive k
  for (int e = threadIdx.x; e < kc * b; e += blockDim.x) {
    const int c = e / kc, kk = e % kc, k = k0 + kk;
    if (c < k) {
      const float v = -__ldg(theta + skew_index(c, k, b));
      if (transposed) dst[c * ld + kk] = v; else dst[kk * ld + c] = v;
    }
  }
}

// Forward.  grid = (b / rows, nb).  Thread e-slots map to (r = e / b, c = e % b).
template <typename OutT>
__global__ void __launch_bounds__(kThreads) cnp_fwd_kernel(const float* __restrict__ theta, int b,
                                                           int n, OutT* __restrict__ Q) {
  extern __shared__ float smem[];
  const int rows = min(kRowSlab, b);
  const int kc = min(kChunk, b);
  const int ldk = b + 1;
  float* cur = smem;                     // [rows][b]  rows of K^m
  float* kch = smem + rows * b;          // [kc][b+1]  rows k0.. of K
  const int j = blockIdx.y;
  const int r0 = blockIdx.x * rows;
  const float* th = theta + (size_t)j * (b * (b - 1) / 2);
  const int nout = rows * b;

  float acc[16], qm[16];   // qm accumulates Q - I
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < nout) {
      const int r = e / b, c = e % b;
      const float k = skew_entry(th, r0 + r, c, b);
      cur[e] = k;
      qm[q] = 2.f * k;   // m = 1 term; n >= 1 so its coefficient is 2
    }
  }
  __syncthreads();
  for (int m = 2; m <= n + 1; ++m) {
    const float coef = (m <= n) ? 2.f : 1.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
    for (int k0 = 0; k0 < b; k0 += kc) {
      stage_skew_rows(th, b, k0, kc, kch, ldk, false);
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int e = threadIdx.x + q * kThreads;
        if (e < nout) {
          const int r = e / b, c = e % b;
          const float* a = cur + r * b + k0;
          float s = acc[q];
          for (int kk = 0; kk < kc; ++kk) s = fmaf(a[kk], kch[kk * ldk + c], s);
          acc[q] = s;
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = threadIdx.x + q * kThreads;
      if (e < nout) {
        cur[e] = acc[q];
        qm[q] = fmaf(coef, acc[q], qm[q]);
      }
    }
    __syncthreads();
  }
  OutT* Qj = Q + (size_t)j * b * b;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < nout) {
      const int r = e / b, c = e % b;
      const float v = qm[q] + ((r0 + r) == c ? 1.f : 0.f);
      Qj[(size_t)(r0 + r) * b + c] = from_f32<OutT>(v);
    }
  }
}

// Backward.  For a column slab of dK, with A = K^T = -K and G = dL/dQ:
//   dK = sum_{a=0}^{n} A^a G p_a(A),  p_a(A) = sum_{c=0}^{n-a} coef_{a+c+1} A^c,
// evaluated by Horner in a (H_n = G, H_a = X_a + A H_{a+1}) while the
// powers grow: with S_c = sum_{i<=c} G A^i,  X_{n-c} = S_{c-1} + S_c.
// Every product is a left multiplication of a column slab, so a CTA needs only
// its own columns.  grid = (b / cols, nb).  e-slots map to (r = e % b, cc = e / b).
__global__ void __launch_bounds__(kThreads) cnp_bwd_kernel(const float* __restrict__ theta,
                                                           const float* __restrict__ dQ, int b,
                                                           int n, float* __restrict__ dtheta) {
  extern __shared__ float smem[];
  const int cols = min(kColSlab, b);
  const int kc = min(kChunk, b);
  const int ldm = kc + 1;
  float* apow = smem;               // [b][cols]  A^c[:, slab]
  float* hs = apow + b * cols;      // [b][cols]  H[:, slab]
  float* mch = hs + b * cols;       // [b][kc+1]  M[:, k0..k0+kc)
  const int j = blockIdx.y;
  const int c0 = blockIdx.x * cols;
  const float* th = theta + (size_t)j * (b * (b - 1) / 2);
  const float* G = dQ + (size_t)j * b * b;
  const int nout = b * cols;

  float sprev[16], acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < nout) {
      const int r = e % b, cc = e / b;
      apow[r * cols + cc] = (r == c0 + cc) ? 1.f : 0.f;
      const float g = G[(size_t)r * b + c0 + cc];
      hs[r * cols + cc] = g;   // H_n = G
      sprev[q] = g;            // S_0 = G A^0
    }
  }
  __syncthreads();

  // acc = M . X[:, slab] with M = A (from theta) or G (from dQ), X in smem.
  auto left_mul = [&](bool m_is_a, const float* X) {
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
    for (int k0 = 0; k0 < b; k0 += kc) {
      if (m_is_a) {
        // A[r][k0+kk] = -K[r][k0+kk] = K[k0+kk][r]: rows of K, stored transposed
        stage_skew_rows(th, b, k0, kc, mch, ldm, true);
      } else {
        for (int e = threadIdx.x; e < b * kc; e += blockDim.x) {
          const int r = e / kc, kk = e % kc;
          mch[r * ldm + kk] = G[(size_t)r * b + k0 + kk];
        }
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int e = threadIdx.x + q * kThreads;
        if (e < nout) {
          const int r = e % b, cc = e / b;
          float s = acc[q];
          for (int kk = 0; kk < kc; ++kk) s = fmaf(mch[r * ldm + kk], X[(k0 + kk) * cols + cc], s);
          acc[q] = s;
        }
      }
      __syncthreads();
    }
  };

  for (int c = 1; c <= n; ++c) {
    left_mul(true, apow);                      // A^c = A . A^{c-1}
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = threadIdx.x + q * kThreads;
      if (e < nout) apow[(e % b) * cols + e / b] = acc[q];
    }
    __syncthreads();
    left_mul(false, apow);                     // G A^c
    float xa[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float scur = sprev[q] + acc[q];    // S_c
      xa[q] = sprev[q] + scur;                 // X_{n-c}
      sprev[q] = scur;
    }
    left_mul(true, hs);                        // A H_{n-c+1}
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = threadIdx.x + q * kThreads;
      if (e < nout) hs[(e % b) * cols + e / b] = xa[q] + acc[q];
    }
    __syncthreads();
  }
  // dtheta(i,k) = dK[i][k] - dK[k][i]: each packed entry receives exactly two
  // contributions onto a zeroed buffer, so the sum is order independent.
  float* dth = dtheta + (size_t)j * (b * (b - 1) / 2);
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < nout) {
      const int r = e % b, c = c0 + e / b;
      const float v = hs[r * cols + e / b];
      if (r < c) atomicAdd(dth + skew_index(r, c, b), v);
      else if (r > c) atomicAdd(dth + skew_index(c, r, b), -v);
    }
  }
}

// Shared-memory layout of the one-CTA-per-block forward: the packed
// parameters, K with a padded row, then H (16-byte aligned).
template <int B>
__host__ __device__ constexpr int small_fwd_h_off() {
  return ((B * (B - 1) / 2 + B * (B + 1)) + 3) / 4 * 4;
}
template <int B>
constexpr size_t small_fwd_smem() {
  return sizeof(float) * ((size_t)small_fwd_h_off<B>() + (size_t)B * B);
}

// Forward for b = 16 (the template takes b up to 128): one CTA holds a whole
// block, K and the running factor in shared memory, and evaluates the
// truncated series in Horner form,
//   H_1 = 2I + K,  H_{s+1} = 2I + K H_s,  Q = I + K H_n
// (= I + 2K + ... + 2K^n + K^{n+1}): n products of b x b.  Each thread owns
// OUT = b*b/256 entries of one row, in groups of four columns 4*TPR apart so
// that the threads of a row read one contiguous row of H per step.
template <int B, typename OutT>
__global__ void __launch_bounds__(kThreads) cnp_fwd_small_kernel(const float* __restrict__ theta,
                                                                 int n, OutT* __restrict__ Q) {
  constexpr int OUT = B * B / kThreads;   // entries per thread: 1, 4, 16, 64
  constexpr int TPR = B / OUT;            // threads per row: 16, 8, 4, 2
  constexpr int NP = B * (B - 1) / 2;
  constexpr int LDK = B + 1;
  extern __shared__ float small_smem[];   // small_fwd_smem<B>() bytes
  float* ths = small_smem;                                 // [NP] packed parameters
  float* Ks = small_smem + small_fwd_h_off<B>() - B * LDK;  // [B][LDK]
  float* Hs = small_smem + small_fwd_h_off<B>();           // [B][B], 16-byte aligned
  const int j = blockIdx.x;
  const float* th = theta + (size_t)j * NP;
  for (int e = threadIdx.x; e < NP; e += kThreads) ths[e] = __ldg(th + e);
  __syncthreads();
  for (int e = threadIdx.x; e < B * B; e += kThreads) {
    const int i = e / B, k = e % B;
    Ks[i * LDK + k] = k > i ? ths[skew_index(i, k, B)] : (k < i ? -ths[skew_index(k, i, B)] : 0.f);
  }
  __syncthreads();
  const int row = threadIdx.x / TPR;
  const int lane_c = threadIdx.x % TPR;
  // column of the thread's entry (q-th group of four, e-th in the group)
  auto col = [&](int q, int e) { return OUT >= 4 ? lane_c * 4 + q * 4 * TPR + e : lane_c; };
  constexpr int NG = OUT >= 4 ? OUT / 4 : 1;   // groups of four
  constexpr int GE = OUT >= 4 ? 4 : 1;         // entries per group
#pragma unroll
  for (int q = 0; q < NG; ++q)
#pragma unroll
    for (int e = 0; e < GE; ++e) {
      const int c = col(q, e);
      Hs[row * B + c] = Ks[row * LDK + c] + (row == c ? 2.f : 0.f);
    }
  __syncthreads();
  float acc[OUT];
  for (int step = 1; step <= n; ++step) {
#pragma unroll
    for (int t = 0; t < OUT; ++t) acc[t] = 0.f;
#pragma unroll 4
    for (int k = 0; k < B; ++k) {
      const float a = Ks[row * LDK + k];
      if constexpr (OUT >= 4) {
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          const float4 h = *reinterpret_cast<const float4*>(Hs + k * B + col(q, 0));
          acc[4 * q + 0] = fmaf(a, h.x, acc[4 * q + 0]);
          acc[4 * q + 1] = fmaf(a, h.y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(a, h.z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(a, h.w, acc[4 * q + 3]);
        }
      } else {
        acc[0] = fmaf(a, Hs[k * B + col(0, 0)], acc[0]);
      }
    }
    if (step < n) {
      __syncthreads();   // every thread is done reading H_s
#pragma unroll
      for (int q = 0; q < NG; ++q)
#pragma unroll
        for (int e = 0; e < GE; ++e) {
          const int c = col(q, e);
          Hs[row * B + c] = acc[q * GE + e] + (row == c ? 2.f : 0.f);
        }
      __syncthreads();
    }
  }
  OutT* qrow = Q + (size_t)j * B * B + (size_t)row * B;
#pragma unroll
  for (int q = 0; q < NG; ++q)
#pragma unroll
    for (int e = 0; e < GE; ++e) {
      const int c = col(q, e);
      qrow[c] = from_f32<OutT>(acc[q * GE + e] + (row == c ? 1.f : 0.f));
    }
}

template <int B>
poetx_status launch_cnp_fwd_small(const float* theta, int nb, int n, void* Q, poetx_dtype out_dtype,
                                  cudaStream_t s) {
  if (nb <= 0) return POETX_OK;
  constexpr size_t smem = small_fwd_smem<B>();
  {
    KernelScope ks_("cnp_fwd_simt", s);
    if (out_dtype == POETX_F32) {
      set_max_dynamic_smem((const void*)cnp_fwd_small_kernel<B, float>, (int)smem);
      cnp_fwd_small_kernel<B, float><<<nb, kThreads, smem, s>>>(theta, n, (float*)Q);
    } else {
      set_max_dynamic_smem((const void*)cnp_fwd_small_kernel<B, __nv_bfloat16>, (int)smem);
      cnp_fwd_small_kernel<B, __nv_bfloat16><<<nb, kThreads, smem, s>>>(theta, n,
                                                                        (__nv_bfloat16*)Q);
    }
  }
  return check_launch();
}

}  // namespace

size_t cnp_fwd_simt_smem(int b) {
  const int rows = b < kRowSlab ? b : kRowSlab;
  const int kc = b < kChunk ? b : kChunk;
  return sizeof(float) * ((size_t)rows * b + (size_t)kc * (b + 1));
}

size_t cnp_bwd_simt_smem(int b) {
  const int cols = b < kColSlab ? b : kColSlab;
  const int kc = b < kChunk ? b : kChunk;
  return sizeof(float) * (2 * (size_t)b * cols + (size_t)b * (kc + 1));
}

poetx_status launch_cnp_fwd_simt(const float* theta, int nb, int b, int n, void* Q,
                                 poetx_dtype out_dtype, cudaStream_t s) {
  // b = 32, 64, 128 take the tensor-core tile kernel (tc_cnp_tile.cu) at any block count
  if (b == 16) return launch_cnp_fwd_small<16>(theta, nb, n, Q, out_dtype, s);
  const int rows = b < kRowSlab ? b : kRowSlab;
  dim3 grid(b / rows, nb);
  const size_t smem = cnp_fwd_simt_smem(b);
  if (out_dtype == POETX_F32) {
    set_max_dynamic_smem((const void*)cnp_fwd_kernel<float>, (int)smem);
    {
      KernelScope ks_("cnp_fwd_simt", s);
      cnp_fwd_kernel<float><<<grid, kThreads, smem, s>>>(theta, b, n, (float*)Q);
    }
  } else {
    set_max_dynamic_smem((const void*)cnp_fwd_kernel<__nv_bfloat16>, (int)smem);
    {
      KernelScope ks_("cnp_fwd_simt", s);
      cnp_fwd_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(theta, b, n, (__nv_bfloat16*)Q);
    }
  }
  return check_launch();
}

namespace {
__global__ void sum_slots_kernel(float* __restrict__ part, int slots, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float acc = part[i];
    for (int s = 1; s < slots; ++s) acc += part[(size_t)s * n + i];
    part[i] = acc;
  }
}
}  // namespace

poetx_status launch_sum_slots(float* part, int slots, size_t n, cudaStream_t s) {
  if (slots <= 1 || n == 0) return POETX_OK;
  const size_t blocks = (n + 255) / 256;
  {
    KernelScope ks_("sum_slots", s);
    sum_slots_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(part, slots, n);
  }
  return check_launch();
}

poetx_status launch_cnp_bwd_simt(const float* theta, const float* dQ, int nb, int b, int n,
                                 float* dtheta, cudaStream_t s) {
  if (cudaMemsetAsync(dtheta, 0, sizeof(float) * (size_t)nb * (b * (b - 1) / 2), s) != cudaSuccess)
    return check_launch();
  const int cols = b < kColSlab ? b : kColSlab;
  dim3 grid(b / cols, nb);
  const size_t smem = cnp_bwd_simt_smem(b);
  set_max_dynamic_smem((const void*)cnp_bwd_kernel, (int)smem);
  {
    KernelScope ks_("cnp_bwd_simt", s);
    cnp_bwd_kernel<<<grid, kThreads, smem, s>>>(theta, dQ, b, n, dtheta);
  }
  return check_launch();
}

}  // namespace poetx
