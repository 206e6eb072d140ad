// linear_simt.cu -- the transformed linear on the CUDA cores (fp32 FFMA).
//
// [POET-X §2.A-§2.C] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, sections 2.A-2.C): the
// layer is applied to the activations as a chain (block-diagonal P, frozen W0,
// block-diagonal R); each block is its own small matrix processed as a batch;
// permutations are index maps applied while loading (gather) or storing
// (scatter).  This file is the exact-fp32 path: it serves fp32 activations
// (any power-of-two block size) and bf16 activations whose block size the
// tensor-core kernels do not take.  Accumulation is always fp32.
#include "common.cuh"
#include "kernels.cuh"
#include "profile.cuh"

namespace poetx {

namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- block apply
// out[t][scat(jb + i)] = sum_k Qop_j[i][k] * in[t][gath(jb + k)]
//   Qop_j = Q_j (transpose_q == 0) or Q_j^T (transpose_q == 1)
//   gath / scat: a permutation array, or NULL for the identity.
// grid = (ceil(T / kTok), d / b); e-slots map to (i = e % b, t = e / b).
constexpr int kTok = 16;
constexpr int kQChunk = 32;

template <typename InT, typename QT, typename OutT>
__global__ void __launch_bounds__(kThreads) block_apply_kernel(
    const InT* __restrict__ in, OutT* __restrict__ out, const QT* __restrict__ Qs, int T, int d,
    int b, const int32_t* __restrict__ gath, const int32_t* __restrict__ scat, int transpose_q) {
  extern __shared__ float smem[];
  const int kc = min(kQChunk, b);
  const int ldq = kc + 1;
  float* xin = smem;                 // [kTok][b]
  float* qch = smem + kTok * b;      // [b][kc+1]  Qop[i][k0 + kk]
  const int t0 = blockIdx.x * kTok;
  const int j = blockIdx.y;
  const int jb = j * b;
  const QT* Q = Qs + (size_t)j * b * b;
  const int ntok = min(kTok, T - t0);

  for (int e = threadIdx.x; e < kTok * b; e += blockDim.x) {
    const int t = e / b, k = e % b;
    float v = 0.f;
    if (t < ntok) {
      const int col = gath ? __ldg(gath + jb + k) : jb + k;
      v = to_f32(in[(size_t)(t0 + t) * d + col]);
    }
    xin[e] = v;
  }
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.f;
  const int nout = kTok * b;
  for (int k0 = 0; k0 < b; k0 += kc) {
    __syncthreads();
    if (!transpose_q) {
      for (int e = threadIdx.x; e < b * kc; e += blockDim.x) {
        const int i = e / kc, kk = e % kc;
        qch[i * ldq + kk] = to_f32(Q[(size_t)i * b + k0 + kk]);
      }
    } else {
      for (int e = threadIdx.x; e < b * kc; e += blockDim.x) {
        const int kk = e / b, i = e % b;
        qch[i * ldq + kk] = to_f32(Q[(size_t)(k0 + kk) * b + i]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = threadIdx.x + q * kThreads;
      if (e < nout) {
        const int i = e % b, t = e / b;
        const float* xr = xin + t * b + k0;
        const float* qr = qch + i * ldq;
        float s = acc[q];
        for (int kk = 0; kk < kc; ++kk) s = fmaf(qr[kk], xr[kk], s);
        acc[q] = s;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < nout) {
      const int i = e % b, t = e / b;
      if (t < ntok) {
        const int col = scat ? __ldg(scat + jb + i) : jb + i;
        out[(size_t)(t0 + t) * d + col] = from_f32<OutT>(acc[q]);
      }
    }
  }
}

// ---------------------------------------------------------------- GEMM
// C[M][N] = sum_k A[M][k] * Bop[k][N]; Bop = B^T with B [N][K] (b_kmajor) or
// B [K][N].  64 x 64 tiles, 16-deep k steps, 4 x 4 outputs per thread.
template <typename T, typename OutT, bool kBKMajor>
__global__ void __launch_bounds__(kThreads) gemm_kernel(const T* __restrict__ A,
                                                        const T* __restrict__ B,
                                                        OutT* __restrict__ C, int M, int N,
                                                        int K) {
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = threadIdx.x; e < 64 * 16; e += kThreads) {
      const int m = e / 16, kk = e % 16;
      const int gm = m0 + m, gk = k0 + kk;
      As[kk][m] = (gm < M && gk < K) ? to_f32(A[(size_t)gm * K + gk]) : 0.f;
    }
    if (kBKMajor) {
      for (int e = threadIdx.x; e < 64 * 16; e += kThreads) {
        const int n = e / 16, kk = e % 16;
        const int gn = n0 + n, gk = k0 + kk;
        Bs[kk][n] = (gn < N && gk < K) ? to_f32(B[(size_t)gn * K + gk]) : 0.f;
      }
    } else {
      for (int e = threadIdx.x; e < 64 * 16; e += kThreads) {
        const int kk = e / 64, n = e % 64;
        const int gn = n0 + n, gk = k0 + kk;
        Bs[kk][n] = (gn < N && gk < K) ? to_f32(B[(size_t)gk * N + gn]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = As[kk][ty * 4 + u];
#pragma unroll
      for (int v = 0; v < 4; ++v) bv[v] = Bs[kk][tx * 4 + v];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int gm = m0 + ty * 4 + u;
    if (gm >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int gn = n0 + tx * 4 + v;
      if (gn < N) C[(size_t)gm * N + gn] = from_f32<OutT>(acc[u][v]);
    }
  }
}

// ---------------------------------------------------------------- dQ token sums
// dQ_j[i][k] += sum_{t in split} G[t][gG(jb+i)] * V[t][gV(jb+k)]   (fp32, atomics)
// grid = (b/32 [k tiles], b/32 [i tiles], nb * splits); 32 x 32 outputs per CTA.
constexpr int kDqTile = 32;
constexpr int kDqTok = 32;

template <typename T>
__global__ void __launch_bounds__(kThreads) dq_kernel(const T* __restrict__ G,
                                                      const T* __restrict__ V, int T_, int d,
                                                      int b, const int32_t* __restrict__ gG,
                                                      const int32_t* __restrict__ gV,
                                                      int tok_per_split, int splits,
                                                      float* __restrict__ dQ) {
  __shared__ float gs[kDqTok][kDqTile + 1];
  __shared__ float vs[kDqTok][kDqTile + 1];
  const int tile = min(kDqTile, b);
  const int k0 = blockIdx.x * tile, i0 = blockIdx.y * tile;
  const int j = blockIdx.z / splits, sp = blockIdx.z % splits;
  const int jb = j * b;
  const int tb = sp * tok_per_split, te = min(T_, tb + tok_per_split);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int t0 = tb; t0 < te; t0 += kDqTok) {
    for (int e = threadIdx.x; e < kDqTok * tile; e += kThreads) {
      const int tt = e / tile, c = e % tile, t = t0 + tt;
      float gv = 0.f, vv = 0.f;
      if (t < te) {
        const int cg = gG ? __ldg(gG + jb + i0 + c) : jb + i0 + c;
        const int cv = gV ? __ldg(gV + jb + k0 + c) : jb + k0 + c;
        gv = to_f32(G[(size_t)t * d + cg]);
        vv = to_f32(V[(size_t)t * d + cv]);
      }
      gs[tt][c] = gv;
      vs[tt][c] = vv;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = threadIdx.x + q * kThreads;
      if (e < tile * tile) {
        const int i = e / tile, k = e % tile;
        float s = acc[q];
        for (int tt = 0; tt < kDqTok; ++tt) s = fmaf(gs[tt][i], vs[tt][k], s);
        acc[q] = s;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = threadIdx.x + q * kThreads;
    if (e < tile * tile) {
      const int i = e / tile, k = e % tile;
      atomicAdd(dQ + ((size_t)j * b + i0 + i) * b + k0 + k, acc[q]);
    }
  }
}

// ---------------------------------------------------------------- permutations
__global__ void invert_perm_kernel(const int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                   int d) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < d) inv[perm[i]] = i;
}

// scratch[0..d) counts hits per value, scratch[d] is the failure flag.
__global__ void perm_count_kernel(const int32_t* __restrict__ perm, int d, int32_t* scratch) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const int32_t v = perm[i];
  if (v < 0 || v >= d) atomicOr(scratch + d, 1);
  else atomicAdd(scratch + v, 1);
}

__global__ void perm_verify_kernel(const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ inv, int d, int32_t* scratch) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  if (scratch[i] != 1) atomicOr(scratch + d, 1);
  if (inv) {
    const int32_t v = perm[i];
    if (v < 0 || v >= d || inv[v] != i) atomicOr(scratch + d, 1);
  }
}

template <typename T>
__global__ void merge_w0_kernel(const T* __restrict__ W0, T* __restrict__ W0m, int d_out,
                                int d_in, const int32_t* __restrict__ po,
                                const int32_t* __restrict__ pi) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (k < d_in) W0m[(size_t)i * d_in + k] = W0[(size_t)__ldg(po + i) * d_in + __ldg(pi + k)];
}

// ---------------------------------------------------------------- transpose
// out[c][r] = in[r][c] for in [rows][cols]: one 32 x 32 tile per CTA of
// 32 x 8 threads, read and written along rows (coalesced) through shared
// memory (a padded column removes bank conflicts).
constexpr int kTr = 32;

template <typename T>
__global__ void __launch_bounds__(kTr * 8) transpose_kernel(const T* __restrict__ in,
                                                            T* __restrict__ out, int rows,
                                                            int cols) {
  __shared__ T tile[kTr][kTr + 1];
  const int c0 = blockIdx.x * kTr, r0 = blockIdx.y * kTr;
  for (int k = threadIdx.y; k < kTr; k += 8) {
    const int r = r0 + k, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[k][threadIdx.x] = in[(size_t)r * cols + c];
  }
  __syncthreads();
  for (int k = threadIdx.y; k < kTr; k += 8) {
    const int c = c0 + k, r = r0 + threadIdx.x;
    if (c < cols && r < rows) out[(size_t)c * rows + r] = tile[threadIdx.x][k];
  }
}

}  // namespace

// ---------------------------------------------------------------- launchers

poetx_status launch_block_apply_simt(const void* in, void* out, const void* Qs, int T, int d,
                                     int b, const int32_t* gath, const int32_t* scat,
                                     bool transpose_q, poetx_dtype dt, cudaStream_t s) {
  if (T <= 0) return POETX_OK;
  dim3 grid((T + kTok - 1) / kTok, d / b);
  const int kc = b < kQChunk ? b : kQChunk;
  const size_t smem = sizeof(float) * ((size_t)kTok * b + (size_t)b * (kc + 1));
  if (dt == POETX_F32) {
    auto k = block_apply_kernel<float, float, float>;
    set_max_dynamic_smem((const void*)k, (int)smem);
    {
      KernelScope ks_("block_apply_simt", s);
      k<<<grid, kThreads, smem, s>>>((const float*)in, (float*)out, (const float*)Qs, T, d, b, gath,
                                     scat, transpose_q ? 1 : 0);
    }
  } else {
    auto k = block_apply_kernel<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>;
    set_max_dynamic_smem((const void*)k, (int)smem);
    {
      KernelScope ks_("block_apply_simt", s);
      k<<<grid, kThreads, smem, s>>>((const __nv_bfloat16*)in, (__nv_bfloat16*)out,
                                     (const __nv_bfloat16*)Qs, T, d, b, gath, scat,
                                     transpose_q ? 1 : 0);
    }
  }
  return check_launch();
}

poetx_status launch_gemm_simt(const void* A, const void* B, void* C, int M, int N, int K,
                              bool b_kmajor, poetx_dtype dt, cudaStream_t s) {
  if (M <= 0 || N <= 0) return POETX_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  if (dt == POETX_F32) {
    if (b_kmajor)
      {
        KernelScope ks_("gemm_simt", s);
        gemm_kernel<float, float, true><<<grid, kThreads, 0, s>>>((const float*)A, (const float*)B,
                                                                  (float*)C, M, N, K);
      }
    else
      {
        KernelScope ks_("gemm_simt", s);
        gemm_kernel<float, float, false><<<grid, kThreads, 0, s>>>((const float*)A, (const float*)B,
                                                                   (float*)C, M, N, K);
      }
  } else {
    using bf = __nv_bfloat16;
    if (b_kmajor)
      {
        KernelScope ks_("gemm_simt", s);
        gemm_kernel<bf, bf, true><<<grid, kThreads, 0, s>>>((const bf*)A, (const bf*)B, (bf*)C, M, N, K);
      }
    else
      {
        KernelScope ks_("gemm_simt", s);
        gemm_kernel<bf, bf, false><<<grid, kThreads, 0, s>>>((const bf*)A, (const bf*)B, (bf*)C, M, N,
                                                             K);
      }
  }
  return check_launch();
}

poetx_status launch_dq_simt(const void* G, const void* V, int T, int d, int b, const int32_t* gG,
                            const int32_t* gV, float* dQ, poetx_dtype dt, cudaStream_t s) {
  if (cudaMemsetAsync(dQ, 0, sizeof(float) * (size_t)d * b, s) != cudaSuccess) return check_launch();
  if (T <= 0) return POETX_OK;
  const int tile = b < kDqTile ? b : kDqTile;
  const int tok_per_split = 512;
  const int splits = (T + tok_per_split - 1) / tok_per_split;
  dim3 grid(b / tile, b / tile, (d / b) * splits);
  if (dt == POETX_F32)
    {
      KernelScope ks_("dq_simt", s);
      dq_kernel<float><<<grid, kThreads, 0, s>>>((const float*)G, (const float*)V, T, d, b, gG, gV,
                                                 tok_per_split, splits, dQ);
    }
  else
    {
      KernelScope ks_("dq_simt", s);
      dq_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>((const __nv_bfloat16*)G,
                                                         (const __nv_bfloat16*)V, T, d, b, gG, gV,
                                                         tok_per_split, splits, dQ);
    }
  return check_launch();
}

poetx_status launch_invert_perm(const int32_t* perm, int32_t* inv, int d, cudaStream_t s) {
  if (d <= 0) return POETX_OK;
  {
    KernelScope ks_("invert_perm", s);
    invert_perm_kernel<<<(d + 255) / 256, 256, 0, s>>>(perm, inv, d);
  }
  return check_launch();
}

poetx_status launch_check_perm(const int32_t* perm, const int32_t* inv, int d, int32_t* scratch,
                               int32_t* flag_host, cudaStream_t s) {
  *flag_host = 0;
  if (d <= 0) return POETX_OK;
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t) * ((size_t)d + 1), s) != cudaSuccess)
    return check_launch();
  {
    KernelScope ks_("check_perm", s);
    perm_count_kernel<<<(d + 255) / 256, 256, 0, s>>>(perm, d, scratch);
  }
  {
    KernelScope ks_("check_perm", s);
    perm_verify_kernel<<<(d + 255) / 256, 256, 0, s>>>(perm, inv, d, scratch);
  }
  if (cudaMemcpyAsync(flag_host, scratch + d, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return check_launch();
  if (cudaStreamSynchronize(s) != cudaSuccess) return check_launch();
  return check_launch();
}

poetx_status launch_merge_w0(const void* W0, void* W0m, int d_out, int d_in, poetx_dtype dt,
                             const int32_t* po, const int32_t* pi, cudaStream_t s) {
  if (d_out <= 0 || d_in <= 0) return POETX_OK;
  dim3 grid((d_in + 255) / 256, d_out);
  if (dt == POETX_F32)
    {
      KernelScope ks_("merge_w0", s);
      merge_w0_kernel<float><<<grid, 256, 0, s>>>((const float*)W0, (float*)W0m, d_out, d_in, po, pi);
    }
  else
    {
      KernelScope ks_("merge_w0", s);
      merge_w0_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)W0,
                                                          (__nv_bfloat16*)W0m, d_out, d_in, po, pi);
    }
  return check_launch();
}

poetx_status launch_transpose(const void* in, void* out, int rows, int cols, poetx_dtype dt,
                              cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return POETX_OK;
  const dim3 grid((cols + kTr - 1) / kTr, (rows + kTr - 1) / kTr), block(kTr, 8);
  if (grid.y > 65535) return POETX_ERR_SHAPE;
  {
    KernelScope ks_("transpose", s);
    if (dt == POETX_F32)
      transpose_kernel<float><<<grid, block, 0, s>>>((const float*)in, (float*)out, rows, cols);
    else
      transpose_kernel<__nv_bfloat16><<<grid, block, 0, s>>>((const __nv_bfloat16*)in,
                                                             (__nv_bfloat16*)out, rows, cols);
  }
  return check_launch();
}

}  // namespace poetx
