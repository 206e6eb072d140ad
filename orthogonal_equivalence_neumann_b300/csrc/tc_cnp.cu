// tc_cnp.cu -- Cayley-Neumann blocks and their backward on the tensor cores.
//
// [POET-X §2.D] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.D): Q = (I + K)(I + K +
// ... + K^n) for skew K stored as its upper triangle; the page fuses the
// Neumann chain in one kernel that keeps K and its powers on chip.
//
// Both directions run the same right-multiplication chain on a slab of 128
// rows, so every CTA (block j, row slab) is independent:
//   forward   X_1 = K,  X_{i+1} = X_i K + 2K,        Q = I + X_{n+1}
//             (Horner form of Q - I = 2K + 2K^2 + ... + 2K^n + K^{n+1})
//   backward  with G = dL/dQ, the adjoint dK = sum_m c_m sum_a (K^T)^a G
//             (K^T)^{m-1-a} is the upper-right block of the same polynomial
//             of [[K^T, G], [0, K^T]], whose top block row follows
//             X_1 = K^T, Y_1 = G,
//             X_{i+1} = X_i K^T + 2K^T,  Y_{i+1} = X_i G + Y_i K^T + 2G,
//             dK = Y_{n+1};  dtheta(i,k) = dK[i][k] - dK[k][i].
// Each step is a tcgen05.mma chain (M = 128 rows, N = b, K = 16, bf16
// operands, fp32 accumulation in TMEM).  The "+2K" / "+2G" terms are added
// in fp32 when a TMEM result becomes the next step's bf16 A operand, so the
// rounding acts on the Horner terms, not on the identity.
//
// Forward: the CTA unpacks K^T once, straight from the packed parameters,
// into shared memory, where it stays as the B operand of every step (the
// dense K never touches HBM).  Backward (inside the layer's backward, which
// has a workspace): a prep kernel writes dense bf16 K and bf16 G per block
// once; the chain kernel streams them in by TMA, both sides (P and R) in one
// launch.  fp32 Q and the fp32 backward entry point use the exact CUDA-core
// kernels.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kSmemMax = 232448;
constexpr int kMaxStages = 4;

__device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ float bf16_at(const uint8_t* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

// ====================================================================== forward
constexpr int kFwdThreads = 288;   // warp 0: TMEM + MMA; warps 1..8: workers
constexpr int kFwdWorkers = 256;

template <int B>
__global__ void __launch_bounds__(kFwdThreads, 1)
    cnp_fwd_kernel(const float* __restrict__ theta, void* __restrict__ out, int out_f32, int n,
                   int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* bres = smem;                  // [B rows c][B k], K-major: element (c, k) = K[k][c]
  uint8_t* amat = smem + B * B * 2;      // X_i, rows [128][B]
  uint64_t* afull = reinterpret_cast<uint64_t*>(amat + 128 * B * 2);
  uint64_t* stepdone = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stepdone + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.y;
  const int r0 = blockIdx.x * 128;
  constexpr int P = B * (B - 1) / 2;
  const float* th = theta + (size_t)j * P;

  if (threadIdx.x == 0) {
    mbar_init(afull, kFwdWorkers);
    mbar_init(stepdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, B);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, B, false, false);
      const uint32_t ab = smem_u32(amat), bb = smem_u32(bres);
      for (int i = 1; i <= n; ++i) {
        if (!mbar_wait(afull, (i - 1) & 1, err)) break;
        tc_fence_after();
#pragma unroll
        for (int kc = 0; kc < B / 64; ++kc)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem_base, sw128_desc(ab + kc * 128 * 128 + kk * 32, 16, 1024),
                     sw128_desc(bb + kc * B * 128 + kk * 32, 16, 1024), idesc, (kc | kk) != 0);
        mma_commit(stepdone);
      }
    }
  } else {
    const int wt = threadIdx.x - 32;
    const int quarter = warp % 4;
    const int half = (warp - 1) / 4;
    const int r = quarter * 32 + lane;
    const int row = r0 + r;
    bool ok = true;
    // ---- K^T into shared memory, once: unit (c, k..k+8) = K[k..k+8][c]
#pragma unroll 4
    for (int u = wt; u < B * B / 8; u += kFwdWorkers) {
      const int c = u % B, k = (u / B) * 8;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = skew_entry(th, k + e, c, B);
      *reinterpret_cast<uint4*>(bres + sw128_offset(c, k, B)) = pack8(v);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kFwdWorkers) : "memory");   // K^T complete
    for (int i = 1; i <= n && ok; ++i) {
      if (i > 1) {
        if (!(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
        tc_fence_after();
      }
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        float x[32];
        if (i == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = bf16_at(bres, sw128_offset(c0 + e, row, B));
        } else {
          uint32_t rr[32];
          tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            x[e] = __uint_as_float(rr[e]) + 2.f * bf16_at(bres, sw128_offset(c0 + e, row, B));
        }
#pragma unroll
        for (int g = 0; g < 4; ++g)
          *reinterpret_cast<uint4*>(amat + sw128_offset(r, c0 + 8 * g, 128)) = pack8(x + 8 * g);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(afull);
    }
    if (ok && mbar_wait(stepdone, (n - 1) & 1, err)) {
      tc_fence_after();
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
        tmem_ld_wait();
        float q[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)   // the last 2K in fp32, from the packed parameters
          q[e] = __uint_as_float(rr[e]) + 2.f * skew_entry(th, row, c0 + e, B) +
                 (row == c0 + e ? 1.f : 0.f);
        if (out_f32) {
          float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + ((size_t)j * B + row) * B + c0);
#pragma unroll
          for (int g = 0; g < 8; ++g) o[g] = make_float4(q[4 * g], q[4 * g + 1], q[4 * g + 2], q[4 * g + 3]);
        } else {
          uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + ((size_t)j * B + row) * B + c0);
#pragma unroll
          for (int g = 0; g < 4; ++g) o[g] = pack8(q + 8 * g);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, B);
  }
}

// ====================================================================== backward
struct Side {
  const float* theta;
  const float* dQ;
  __nv_bfloat16* Kd;   // dense K, [nb, b, b] bf16
  __nv_bfloat16* Gd;   // dQ in bf16, [nb, b, b]
  float* dtheta;
  int nb, b;
};

// Kd[j][c][k] = bf16(K_j[c][k]), Gd[j][c][k] = bf16(dQ_j[c][k]) for both sides.
__global__ void cnp_prep_kernel(Side sp, Side sr) {
  const bool is_r = (int)blockIdx.y >= sp.nb;
  const Side& sd = is_r ? sr : sp;
  const int j = is_r ? (int)blockIdx.y - sp.nb : (int)blockIdx.y;
  const int b = sd.b;
  const int u = blockIdx.x * blockDim.x + threadIdx.x;   // unit: row c, 8 consecutive k
  if (u >= b * b / 8) return;
  const int c = u / (b / 8), k = (u % (b / 8)) * 8;
  const float* th = sd.theta + (size_t)j * (b * (b - 1) / 2);
  const float* g = sd.dQ + ((size_t)j * b + c) * b + k;
  float kv[8], gv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    kv[e] = skew_entry(th, c, k + e, b);
    gv[e] = g[e];
  }
  *reinterpret_cast<uint4*>(sd.Kd + ((size_t)j * b + c) * b + k) = pack8(kv);
  *reinterpret_cast<uint4*>(sd.Gd + ((size_t)j * b + c) * b + k) = pack8(gv);
}

constexpr int kBwdThreads = 320;   // warp 0: TMEM + MMA; warp 1: TMA; warps 2..9: workers
constexpr int kBwdWorkers = 256;

__global__ void __launch_bounds__(kBwdThreads, 1)
    cnp_bwd_kernel(const __grid_constant__ CUtensorMap tkP, const __grid_constant__ CUtensorMap tgP,
                   const __grid_constant__ CUtensorMap tkR, const __grid_constant__ CUtensorMap tgR,
                   Side sp, Side sr, int n, int bmax, int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const bool is_r = (int)blockIdx.y >= sp.nb;
  const Side& sd = is_r ? sr : sp;
  const CUtensorMap* tk = is_r ? &tkR : &tkP;
  const CUtensorMap* tg = is_r ? &tgR : &tgP;
  const int j = is_r ? (int)blockIdx.y - sp.nb : (int)blockIdx.y;
  const int b = sd.b;
  if ((int)blockIdx.x * 128 >= b) return;    // row slabs exist up to the larger block size
  const int r0 = blockIdx.x * 128;
  const int a_bytes = 128 * bmax * 2;
  const int chunk_bytes = bmax * 64 * 2;
  uint8_t* ax = smem;
  uint8_t* ay = smem + a_bytes;
  uint8_t* ring = smem + 2 * a_bytes;
  uint64_t* bfull = reinterpret_cast<uint64_t*>(ring + stages * chunk_bytes);
  uint64_t* bempty = bfull + kMaxStages;
  uint64_t* afull = bempty + kMaxStages;
  uint64_t* stepdone = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stepdone + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kchunks = b / 64;
  const uint32_t ncols = (uint32_t)(2 * b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bfull + s, 1);
      mbar_init(bempty + s, 1);
    }
    mbar_init(afull, kBwdWorkers);
    mbar_init(stepdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 1) {
    // ------------------------------------------------ TMA: per step, K chunks then G^T chunks
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 1; i <= n && ok; ++i)
        for (int c = 0; c < 2 * kchunks && ok; ++c) {
          if (!(ok = mbar_wait(bempty + st, ph ^ 1, err))) break;
          mbar_arrive_expect_tx(bfull + st, (uint32_t)(b * 128));
          uint8_t* dst = ring + st * chunk_bytes;
          if (c < kchunks) {
            tma_load_2d(dst, tk, c * 64, j * b, bfull + st);           // B[cc][k] = K[cc][k]
          } else {
            const int kc = c - kchunks;
            for (int q = 0; q < b / 64; ++q)                          // B[cc][k] = G[k][cc]
              tma_load_2d(dst + q * 8192, tg, q * 64, j * b + kc * 64, bfull + st);
          }
          if (++st == stages) { st = 0; ph ^= 1; }
        }
    }
  } else if (warp == 0) {
    // ------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t idk = idesc_bf16(128, b, false, false);
      const uint32_t idg = idesc_bf16(128, b, false, true);
      const uint32_t dx = tmem_base, dy = tmem_base + (uint32_t)b;
      const uint32_t axb = smem_u32(ax), ayb = smem_u32(ay);
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 1; i <= n && ok; ++i) {
        if (!(ok = mbar_wait(afull, (i - 1) & 1, err))) break;
        tc_fence_after();
        for (int c = 0; c < 2 * kchunks && ok; ++c) {
          if (!(ok = mbar_wait(bfull + st, ph, err))) break;
          tc_fence_after();
          const uint32_t bb = smem_u32(ring + st * chunk_bytes);
          const int kc = c % kchunks;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t xdesc = sw128_desc(axb + kc * 128 * 128 + kk * 32, 16, 1024);
            if (c < kchunks) {
              const uint64_t bdesc = sw128_desc(bb + kk * 32, 16, 1024);
              const uint32_t acc = (kc | kk) != 0;
              if (i < n) mma_bf16(dx, xdesc, bdesc, idk, acc);                    // X K^T
              mma_bf16(dy, sw128_desc(ayb + kc * 128 * 128 + kk * 32, 16, 1024), bdesc, idk,
                       acc);                                                    // Y K^T
            } else {
              mma_bf16(dy, xdesc, sw128_desc(bb + kk * 2048, 8192, 1024), idg, 1);  // X G
            }
          }
          mma_commit(bempty + st);
          if (++st == stages) { st = 0; ph ^= 1; }
        }
        mma_commit(stepdone);
      }
    }
  } else {
    // ------------------------------------------------ workers: A operands and dtheta
    const int quarter = warp % 4;
    const int half = (warp - 2) / 4;
    const int r = quarter * 32 + lane;
    const int row = r0 + r;
    const __nv_bfloat16* krow = sd.Kd + ((size_t)j * b + row) * b;   // K[row][.]
    const float* grow = sd.dQ + ((size_t)j * b + row) * b;           // G[row][.]
    bool ok = true;
    for (int i = 1; i <= n && ok; ++i) {
      if (i > 1) {
        if (!(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
        tc_fence_after();
      }
      for (int c0 = half * (b / 2); c0 < (half + 1) * (b / 2); c0 += 32) {
        float x[32], y[32];
        if (i == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = -__bfloat162float(krow[c0 + e]);   // K^T[row][c] = -K[row][c]
            y[e] = grow[c0 + e];
          }
        } else {
          uint32_t rx[32], ry[32];
          tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rx);
          tmem_ld32(tmem_base + (uint32_t)(b + c0) + ((uint32_t)(quarter * 32) << 16), ry);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(rx[e]) - 2.f * __bfloat162float(krow[c0 + e]);
            y[e] = __uint_as_float(ry[e]) + 2.f * grow[c0 + e];
          }
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          *reinterpret_cast<uint4*>(ax + sw128_offset(r, c0 + 8 * g, 128)) = pack8(x + 8 * g);
          *reinterpret_cast<uint4*>(ay + sw128_offset(r, c0 + 8 * g, 128)) = pack8(y + 8 * g);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(afull);
    }
    if (ok && mbar_wait(stepdone, (n - 1) & 1, err)) {
      tc_fence_after();
      float* dth = sd.dtheta + (size_t)j * (b * (b - 1) / 2);
      for (int c0 = half * (b / 2); c0 < (half + 1) * (b / 2); c0 += 32) {
        uint32_t ry[32];
        tmem_ld32(tmem_base + (uint32_t)(b + c0) + ((uint32_t)(quarter * 32) << 16), ry);
        tmem_ld_wait();
        // dK = Y_{n+1}; each packed entry receives exactly two adds onto a zeroed buffer
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int c = c0 + e;
          const float v = __uint_as_float(ry[e]) + 2.f * grow[c];
          if (row < c) atomicAdd(dth + skew_index(row, c, b), v);
          else if (row > c) atomicAdd(dth + skew_index(c, row, b), -v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ncols);
  }
}

}  // namespace

bool cnp_supported(int b) { return b == 128 || b == 256; }

poetx_status cnp_fwd_bf16ops(const float* theta, int nb, int b, int n, void* Q, bool out_f32,
                             cudaStream_t s) {
  if (nb <= 0) return POETX_OK;
  if (!cnp_supported(b) || n < 1 || nb > 65535) return POETX_ERR_UNSUPPORTED;
  const int smem = b * b * 2 + 128 * b * 2 + 1024 + 256;
  dim3 grid(b / 128, nb);
  int* err = device_error_word();
  KernelScope ks_("tc_cnp_fwd", s);
  if (b == 256) {
    cudaFuncSetAttribute(cnp_fwd_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cnp_fwd_kernel<256><<<grid, kFwdThreads, smem, s>>>(theta, Q, out_f32 ? 1 : 0, n, err);
  } else {
    cudaFuncSetAttribute(cnp_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cnp_fwd_kernel<128><<<grid, kFwdThreads, smem, s>>>(theta, Q, out_f32 ? 1 : 0, n, err);
  }
  return check_launch();
}

size_t cnp_bwd_workspace_bytes(int d_in, int b_in, int d_out, int b_out) {
  // dense bf16 K and bf16 G for every block of both sides
  return 2 * 2 * ((size_t)d_in * b_in + (size_t)d_out * b_out);
}

poetx_status cnp_bwd_layer(const float* theta_P, const float* dQ_P, int nb_P, int b_P,
                           const float* theta_R, const float* dQ_R, int nb_R, int b_R, int n,
                           float* dtheta_P, float* dtheta_R, void* ws, cudaStream_t s) {
  if (!cnp_supported(b_P) || !cnp_supported(b_R) || n < 1 || nb_P + nb_R > 65535)
    return POETX_ERR_UNSUPPORTED;
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(ws);
  Side sp{theta_P, dQ_P, w, w + (size_t)nb_P * b_P * b_P, dtheta_P, nb_P, b_P};
  __nv_bfloat16* w2 = w + 2 * (size_t)nb_P * b_P * b_P;
  Side sr{theta_R, dQ_R, w2, w2 + (size_t)nb_R * b_R * b_R, dtheta_R, nb_R, b_R};
  if (cudaMemsetAsync(dtheta_P, 0, sizeof(float) * (size_t)nb_P * (b_P * (b_P - 1) / 2), s) !=
          cudaSuccess ||
      cudaMemsetAsync(dtheta_R, 0, sizeof(float) * (size_t)nb_R * (b_R * (b_R - 1) / 2), s) !=
          cudaSuccess)
    return check_launch();
  const int bmax = b_P > b_R ? b_P : b_R;
  {
    dim3 grid((bmax * bmax / 8 + 255) / 256, nb_P + nb_R);
    KernelScope ks_("tc_cnp_bwd_prep", s);
    cnp_prep_kernel<<<grid, 256, 0, s>>>(sp, sr);
  }
  const poetx_status st = check_launch();
  if (st != POETX_OK) return st;
  CUtensorMap tkP, tgP, tkR, tgR;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_2d(&tkP, sp.Kd, bf, 2, (uint64_t)nb_P * b_P, (uint64_t)b_P, (uint32_t)b_P, 64, sw) ||
      !make_tmap_2d(&tgP, sp.Gd, bf, 2, (uint64_t)nb_P * b_P, (uint64_t)b_P, 64, 64, sw) ||
      !make_tmap_2d(&tkR, sr.Kd, bf, 2, (uint64_t)nb_R * b_R, (uint64_t)b_R, (uint32_t)b_R, 64, sw) ||
      !make_tmap_2d(&tgR, sr.Gd, bf, 2, (uint64_t)nb_R * b_R, (uint64_t)b_R, 64, 64, sw))
    return POETX_ERR_CUDA;
  const int a_bytes = 128 * bmax * 2, chunk_bytes = bmax * 64 * 2;
  int stages = (kSmemMax - 2 * a_bytes - 1024 - 256) / chunk_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  const int smem = 2 * a_bytes + stages * chunk_bytes + 1024 + 256;
  cudaFuncSetAttribute(cnp_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  dim3 grid(bmax / 128, nb_P + nb_R);
  {
    KernelScope ks_("tc_cnp_bwd", s);
    cnp_bwd_kernel<<<grid, kBwdThreads, smem, s>>>(tkP, tgP, tkR, tgR, sp, sr, n, bmax, stages,
                                                   device_error_word());
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
