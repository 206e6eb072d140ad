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
// Each step is one tcgen05.mma chain (M = 128 rows, N = b, K = 16) into TMEM
// (X, and Y for the backward: 2 x b fp32 columns).  The "+2K" / "+2G" terms
// are added exactly in fp32 when a TMEM result becomes the next step's bf16
// A operand, so rounding acts only on the small Horner terms.  B operands
// (K, K^T or G^T, 64 columns of k at a time) are unpacked by the worker warps
// straight from the packed parameters (or from dQ) into a shared-memory ring;
// the dense K never touches HBM.
//
// Operands are bf16 (fp32 accumulation): used for bf16 Q and for the backward
// of the bf16 layer.  fp32 Q and the fp32 backward entry point use the exact
// CUDA-core kernels.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kThreads = 288;   // warp 0: TMEM + MMA; warps 1..8: workers
constexpr int kWorkers = 256;
constexpr int kSmemMax = 232448;
constexpr int kMaxStages = 6;

__device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows) {
  return (uint32_t)((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

struct Plan {
  int a_bytes;      // one A operand: 128 rows x b, bf16
  int chunk_bytes;  // one B chunk: b rows x 64 k, bf16
  int stages;
  int smem;
};

Plan plan(int b, bool bwd) {
  Plan p;
  p.a_bytes = 128 * b * 2;
  p.chunk_bytes = b * 64 * 2;
  const int fixed = (bwd ? 2 : 1) * p.a_bytes + 1024 + 256;
  p.stages = (kSmemMax - fixed) / p.chunk_bytes;
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  p.smem = fixed + p.stages * p.chunk_bytes;
  return p;
}

template <bool BWD>
__global__ void __launch_bounds__(kThreads, 1)
    cnp_kernel(const float* __restrict__ theta, const float* __restrict__ dQ, void* __restrict__ out,
               int out_f32, int b, int n, int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int a_bytes = 128 * b * 2;
  const int chunk_bytes = b * 64 * 2;
  uint8_t* ax = smem;
  uint8_t* ay = smem + a_bytes;                          // backward only
  uint8_t* ring = smem + (BWD ? 2 : 1) * a_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + stages * chunk_bytes);
  uint64_t* bfull = bars;
  uint64_t* bempty = bfull + kMaxStages;
  uint64_t* afull = bempty + kMaxStages;
  uint64_t* stepdone = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stepdone + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j = blockIdx.y;
  const int r0 = blockIdx.x * 128;
  const int p = b * (b - 1) / 2;
  const float* th = theta + (size_t)j * p;
  const float* G = BWD ? dQ + (size_t)j * b * b : nullptr;
  const int kchunks = b / 64;
  const uint32_t ncols = (uint32_t)(BWD ? 2 * b : b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bfull + s, kWorkers);
      mbar_init(bempty + s, 1);
    }
    mbar_init(afull, kWorkers);
    mbar_init(stepdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, b, false, false);
      const uint32_t dx = tmem_base, dy = tmem_base + (uint32_t)b;
      int st = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 1; i <= n && ok; ++i) {
        if (!(ok = mbar_wait(afull, (i - 1) & 1, err))) break;
        tc_fence_after();
        const uint32_t axb = smem_u32(ax), ayb = smem_u32(ay);
        const int nchunks = BWD ? 2 * kchunks : kchunks;
        for (int c = 0; c < nchunks && ok; ++c) {
          if (!(ok = mbar_wait(bfull + st, ph, err))) break;
          tc_fence_after();
          const uint32_t bb = smem_u32(ring + st * chunk_bytes);
          const int kc = c % kchunks;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(bb + kk * 32, 16, 1024);
            const uint64_t xdesc = sw128_desc(axb + kc * 128 * 128 + kk * 32, 16, 1024);
            const uint32_t first = (kc | kk) == 0;
            if (!BWD) {
              mma_bf16(dx, xdesc, bdesc, idesc, !first);          // X K
            } else if (c < kchunks) {                             // B = K chunk
              if (i < n) mma_bf16(dx, xdesc, bdesc, idesc, !first);   // X K^T
              const uint64_t ydesc = sw128_desc(ayb + kc * 128 * 128 + kk * 32, 16, 1024);
              mma_bf16(dy, ydesc, bdesc, idesc, !first);          // Y K^T
            } else {                                              // B = G^T chunk
              mma_bf16(dy, xdesc, bdesc, idesc, 1);               // X G
            }
          }
          mma_commit(bempty + st);
          if (++st == stages) { st = 0; ph ^= 1; }
        }
        mma_commit(stepdone);
      }
    }
  } else {
    // ------------------------------------------------------------ workers
    const int wt = threadIdx.x - 32;          // 0..255
    const int quarter = warp % 4;
    const int half = (warp - 1) / 4;          // which half of the columns this warp converts
    const int r = quarter * 32 + lane;        // row within the slab (TMEM lane)
    const int row = r0 + r;                   // row within the block
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    // K-term of the chain: forward K[row][c], backward K^T[row][c] = -K[row][c]
    auto kterm = [&](int c) -> float {
      const float v = skew_entry(th, row, c, b);
      return BWD ? -v : v;
    };
    for (int i = 1; i <= n && ok; ++i) {
      // ---- A operands of step i: X_i (and Y_i) as bf16, 128-byte swizzled
      if (i > 1 && !(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
      if (i > 1) tc_fence_after();
      for (int c0 = half * (b / 2); c0 < (half + 1) * (b / 2); c0 += 32) {
        float vx[32], vy[32];
        if (i == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) vx[e] = kterm(c0 + e);
          if (BWD) {
#pragma unroll
            for (int e = 0; e < 32; ++e) vy[e] = G[(size_t)row * b + c0 + e];
          }
        } else {
          uint32_t rr[32];
          tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) vx[e] = __uint_as_float(rr[e]) + 2.f * kterm(c0 + e);
          if (BWD) {
            tmem_ld32(tmem_base + (uint32_t)(b + c0) + ((uint32_t)(quarter * 32) << 16), rr);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              vy[e] = __uint_as_float(rr[e]) + 2.f * G[(size_t)row * b + c0 + e];
          }
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          *reinterpret_cast<uint4*>(ax + sw128_offset(r, c0 + 8 * g, 128)) =
              make_uint4(pack_bf16x2(vx[8 * g], vx[8 * g + 1]), pack_bf16x2(vx[8 * g + 2], vx[8 * g + 3]),
                         pack_bf16x2(vx[8 * g + 4], vx[8 * g + 5]), pack_bf16x2(vx[8 * g + 6], vx[8 * g + 7]));
          if (BWD)
            *reinterpret_cast<uint4*>(ay + sw128_offset(r, c0 + 8 * g, 128)) =
                make_uint4(pack_bf16x2(vy[8 * g], vy[8 * g + 1]), pack_bf16x2(vy[8 * g + 2], vy[8 * g + 3]),
                           pack_bf16x2(vy[8 * g + 4], vy[8 * g + 5]), pack_bf16x2(vy[8 * g + 6], vy[8 * g + 7]));
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(afull);
      // ---- B chunks of step i
      const int nchunks = BWD ? 2 * kchunks : kchunks;
      for (int c = 0; c < nchunks && ok; ++c) {
        if (!(ok = mbar_wait(bempty + st, ph ^ 1, err))) break;
        uint8_t* dst = ring + st * chunk_bytes;
        const int kc = c % kchunks;
        const bool gchunk = BWD && c >= kchunks;
        for (int u = wt; u < b * 8; u += kWorkers) {
          const int cc = u % b, k8 = u / b;       // B row cc, k = kc*64 + 8*k8 .. +8
          const int k = kc * 64 + k8 * 8;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (gchunk) v[e] = G[(size_t)(k + e) * b + cc];        // G^T[cc][k]
            else if (BWD) v[e] = skew_entry(th, cc, k + e, b);     // K[cc][k]
            else v[e] = skew_entry(th, k + e, cc, b);              // K^T... B[cc][k] = K[k][cc]
          }
          *reinterpret_cast<uint4*>(dst + sw128_offset(cc, k8 * 8, b)) =
              make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                         pack_bf16x2(v[6], v[7]));
        }
        fence_proxy_async_smem();
        mbar_arrive(bfull + st);
        if (++st == stages) { st = 0; ph ^= 1; }
      }
    }
    // ---- result of the last step
    if (ok && mbar_wait(stepdone, (n - 1) & 1, err)) {
      tc_fence_after();
      for (int c0 = half * (b / 2); c0 < (half + 1) * (b / 2); c0 += 32) {
        uint32_t rr[32];
        if (!BWD) {
          tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
          tmem_ld_wait();
          float q[32];
#pragma unroll
          for (int e = 0; e < 32; ++e)
            q[e] = __uint_as_float(rr[e]) + 2.f * kterm(c0 + e) + (row == c0 + e ? 1.f : 0.f);
          if (out_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) +
                                                  ((size_t)j * b + row) * b + c0);
#pragma unroll
            for (int g = 0; g < 8; ++g) o[g] = make_float4(q[4 * g], q[4 * g + 1], q[4 * g + 2], q[4 * g + 3]);
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) +
                                                ((size_t)j * b + row) * b + c0);
#pragma unroll
            for (int g = 0; g < 4; ++g)
              o[g] = make_uint4(pack_bf16x2(q[8 * g], q[8 * g + 1]), pack_bf16x2(q[8 * g + 2], q[8 * g + 3]),
                                pack_bf16x2(q[8 * g + 4], q[8 * g + 5]), pack_bf16x2(q[8 * g + 6], q[8 * g + 7]));
          }
        } else {
          tmem_ld32(tmem_base + (uint32_t)(b + c0) + ((uint32_t)(quarter * 32) << 16), rr);
          tmem_ld_wait();
          float* dth = static_cast<float*>(out) + (size_t)j * p;
          // each packed entry receives exactly two adds onto a zeroed buffer
#pragma unroll 4
          for (int e = 0; e < 32; ++e) {
            const int c = c0 + e;
            const float v = __uint_as_float(rr[e]) + 2.f * G[(size_t)row * b + c];
            if (row < c) atomicAdd(dth + skew_index(row, c, b), v);
            else if (row > c) atomicAdd(dth + skew_index(c, row, b), -v);
          }
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
  const Plan pl = plan(b, false);
  cudaFuncSetAttribute(cnp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  dim3 grid(b / 128, nb);
  {
    KernelScope ks_("tc_cnp_fwd", s);
    cnp_kernel<false><<<grid, kThreads, pl.smem, s>>>(theta, nullptr, Q, out_f32 ? 1 : 0, b, n,
                                                      pl.stages, device_error_word());
  }
  return check_launch();
}

poetx_status cnp_bwd_bf16ops(const float* theta, const float* dQ, int nb, int b, int n,
                             float* dtheta, cudaStream_t s) {
  if (nb <= 0) return POETX_OK;
  if (!cnp_supported(b) || n < 1 || nb > 65535) return POETX_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(dtheta, 0, sizeof(float) * (size_t)nb * (b * (b - 1) / 2), s) != cudaSuccess)
    return check_launch();
  const Plan pl = plan(b, true);
  cudaFuncSetAttribute(cnp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  dim3 grid(b / 128, nb);
  {
    KernelScope ks_("tc_cnp_bwd", s);
    cnp_kernel<true><<<grid, kThreads, pl.smem, s>>>(theta, dQ, dtheta, 1, b, n, pl.stages,
                                                     device_error_word());
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
