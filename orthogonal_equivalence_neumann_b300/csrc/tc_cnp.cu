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
#include <cuda_fp16.h>

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


// ====================================================================== forward
constexpr int kFwdThreads = 288;   // warp 0: TMEM + MMA; warps 1..8: workers
constexpr int kFwdWorkers = 256;

// First packed index of row i (entries (i, i+1) .. (i, b-1)).
__device__ __forceinline__ int skew_row_start(int i, int b) { return (i * (2 * b - i - 1)) >> 1; }

// 8 bf16 of a 16-byte shared-memory unit, widened.
__device__ __forceinline__ void ld_bf16x8(const uint8_t* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// Two parameter sets (the P and R factors of a layer) may share a launch:
// blockIdx.y < nb0 selects the first, the rest the second.
struct FwdSide {
  const float* theta;
  void* Q;
  int nb;
};

constexpr int kUnpackThreads = 256;
constexpr int kUnpackRows = 32;

// Writes Kop = -K (bf16, row-major) of every block into the block's own Q
// buffer, which the chain kernel then loads by TMA and finally overwrites
// with Q.  One CTA per 32-row group of one block; the rows are assembled in
// shared memory (row pitch B + 2 halves, so the column writes fall in
// distinct banks): Kop[c][k] = -theta(c, k) right of the diagonal (packed row
// c), +theta(k, c) left of it (packed rows k hold the group's columns
// contiguously).  All loads are issued before the stores that use them.
template <int B>
__global__ void __launch_bounds__(kUnpackThreads)
    cnp_unpack_kernel(FwdSide f0, FwdSide f1) {
  __shared__ __nv_bfloat16 tile[kUnpackRows * (B + 2)];
  constexpr int LD = B + 2;
  constexpr int P = B * (B - 1) / 2;
  const bool second = (int)blockIdx.y >= f0.nb;
  const FwdSide& sd = second ? f1 : f0;
  const int j = second ? (int)blockIdx.y - f0.nb : (int)blockIdx.y;
  const int c0 = blockIdx.x * kUnpackRows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* th = sd.theta + (size_t)j * P;
  constexpr int W = kUnpackThreads / 32;
  // right of the diagonal (and the diagonal): warp w takes rows c0 + w, c0 + w + 8, ...
#pragma unroll
  for (int rr0 = 0; rr0 < kUnpackRows; rr0 += W) {
    const int rr = rr0 + warp, c = c0 + rr;
    const float* prow = th + skew_row_start(c, B) - (c + 1);   // prow[k] = theta(c, k)
    float v[B / 32];
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      v[q] = k > c ? __ldg(prow + k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      if (k >= c) tile[rr * LD + k] = __float2bfloat16_rn(-v[q]);
    }
  }
  // left of the diagonal: lane = row c0 + lane, warp w takes packed rows k = w, w + 8, ...
  {
    const int c = c0 + lane;
    constexpr int U = 8;
    for (int k0 = warp; k0 < c0 + kUnpackRows - 1; k0 += W * U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        v[u] = k < c ? __ldg(th + skew_row_start(k, B) + (c - k - 1)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        if (k < c) tile[lane * LD + k] = __float2bfloat16_rn(v[u]);
      }
    }
  }
  __syncthreads();
  uint32_t* kd = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(sd.Q) + ((size_t)j * B + c0) * B);
  for (int u = threadIdx.x; u < kUnpackRows * B / 2; u += kUnpackThreads) {
    const int r = u / (B / 2), c2 = (u % (B / 2)) * 2;
    kd[u] = *reinterpret_cast<const uint32_t*>(tile + r * LD + c2);
  }
}

// One CTA = one 128-row slab of one block; for B = 256 the two slabs of a
// block form a cluster.  Kop (the MMA B operand of X -> X K: Kop[c][k] =
// K[k][c] = -K[c][k], K-major) arrives by TMA from the block's Q buffer,
// where the unpack kernel left it; once every slab of the block holds it
// (cluster barrier) the buffer may be overwritten with Q.  The steps
//   X_1 = K,  X_{i+1} = X_i K + 2K,  Q = I + X_n K + 2K
// add 2K from the same bf16 operand (the output is bf16); the first step's A
// is the slab's rows of Kop itself, negated by the instruction.
template <int B>
__global__ void __launch_bounds__(kFwdThreads, 1)
    cnp_fwd_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tk1,
                   FwdSide f0, FwdSide f1, int n, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kop = smem;                 // [B rows c][B k] bf16, 128-byte swizzle
  uint8_t* amat = smem + B * B * 2;    // [128 rows][B k] bf16
  uint64_t* afull = reinterpret_cast<uint64_t*>(amat + 128 * B * 2);
  uint64_t* stepdone = afull + 1;
  uint64_t* kfull = stepdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kfull + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool second = (int)blockIdx.y >= f0.nb;
  const int j = second ? (int)blockIdx.y - f0.nb : (int)blockIdx.y;
  void* __restrict__ out = second ? f1.Q : f0.Q;
  const CUtensorMap* tk = second ? &tk1 : &tk0;
  const int r0 = blockIdx.x * 128;

  if (threadIdx.x == 0) {
    mbar_init(afull, kFwdWorkers);
    mbar_init(stepdone, 1);
    mbar_init(kfull, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(kfull, (uint32_t)(B * B * 2));
    for (int q = 0; q < B / 64; ++q) tma_load_2d(kop + q * (B * 128), tk, q * 64, j * B, kfull);
  }
  if (warp == 0) tmem_alloc(tmem_slot, B);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = mbar_wait(kfull, 0, err);
  // every slab of the block holds Kop: the Q buffer may now be overwritten
  if constexpr (B == 256) cluster_sync();

  if (warp == 0) {
    if (lane == 0 && ok) {
      const uint32_t idesc = idesc_bf16(128, B, false, false);
      const uint32_t ab = smem_u32(amat), bb = smem_u32(kop);
      for (int i = 1; i <= n; ++i) {
        if (!mbar_wait(afull, (i - 1) & 1, err)) break;
        tc_fence_after();
        // step 1: A = X_1 = K = -Kop on the slab rows, read from Kop itself
        // with the instruction's negate-A bit (bit 13)
        const uint32_t a0 = i == 1 ? bb + (uint32_t)r0 * 128 : ab;
        const uint32_t a_chunk = i == 1 ? B * 128 : 128 * 128;
        const uint32_t id = i == 1 ? (idesc | (1u << 13)) : idesc;
#pragma unroll
        for (int kc = 0; kc < B / 64; ++kc)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem_base, sw128_desc(a0 + kc * a_chunk + kk * 32, 16, 1024),
                     sw128_desc(bb + kc * B * 128 + kk * 32, 16, 1024), id, (kc | kk) != 0);
        mma_commit(stepdone);
      }
    }
  } else if (ok) {
    const int quarter = warp % 4;
    const int half = (warp - 1) / 4;
    const int r = quarter * 32 + lane;
    const int row = r0 + r;
    // X_1 = K needs no copy: the first products read it from Kop (negated)
    mbar_arrive(afull);
    // ---- X_{i+1} = X_i K + 2K (as the next A operand), and finally Q = I + X_n K + 2K
    for (int i = 2; i <= n + 1 && ok; ++i) {
      if (!(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
      tc_fence_after();
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
        float kr[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) ld_bf16x8(kop + sw128_offset(row, c0 + 8 * g, B), kr + 8 * g);
        tmem_ld_wait();
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(rr[e]) - 2.f * kr[e];   // K = -Kop
        if (i <= n) {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(amat + sw128_offset(r, c0 + 8 * g, 128)) = pack8(x + 8 * g);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (row == c0 + e) x[e] += 1.f;
          uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + ((size_t)j * B + row) * B + c0);
#pragma unroll
          for (int g = 0; g < 4; ++g) o[g] = pack8(x + 8 * g);
        }
      }
      if (i <= n) {
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(afull);
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

// fp32 Q at b = 256 (the three-term split on the tensor cores): the unpack
// writes Kop = -K as two fp16 parts, hi = fp16(Kop), lo = fp16(Kop - hi), into
// the block's own fp32 Q buffer, which holds exactly both: viewed as 16-bit
// [nb * 512][256], block j's hi rows are j * 512 + c and its lo rows
// j * 512 + 256 + c.  (fp16 parts keep 22 significant bits where bf16 parts
// would keep 16: at sigma = 0.05 the bf16 split left rows of Q about 1e-5 off,
// at the fp32 bar; the lo parts of small entries fall into fp16's subnormal
// range, about 3e-8 absolute, far below that bar relative to Q.)  One CTA per 32-row group of one block, the rows
// assembled in fp32 in shared memory (row pitch 257 words: the column writes
// fall in distinct banks); all loads are issued before their stores.
constexpr int kSplitRows = 32;

// Two fp32 values as fp16 hi parts and fp16 lo parts (x = hi + lo + e,
// |e| <= 2^-22 |x| above fp16's subnormal range), each pair packed low first.
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half ha = __float2half_rn(a), hb = __float2half_rn(b);
  const __half la = __float2half_rn(a - __half2float(ha)), lb = __float2half_rn(b - __half2float(hb));
  hi = (uint32_t)__half_as_ushort(ha) | ((uint32_t)__half_as_ushort(hb) << 16);
  lo = (uint32_t)__half_as_ushort(la) | ((uint32_t)__half_as_ushort(lb) << 16);
}

__global__ void __launch_bounds__(kUnpackThreads)
    cnp_unpack_split_kernel(FwdSide f0, FwdSide f1) {
  constexpr int B = 256, LD = B + 1, P = B * (B - 1) / 2;
  __shared__ float tile[kSplitRows * LD];
  const bool second = (int)blockIdx.y >= f0.nb;
  const FwdSide& sd = second ? f1 : f0;
  const int j = second ? (int)blockIdx.y - f0.nb : (int)blockIdx.y;
  const int c0 = blockIdx.x * kSplitRows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* th = sd.theta + (size_t)j * P;
  constexpr int W = kUnpackThreads / 32;
  // right of the diagonal (and the diagonal): warp w takes rows c0 + w, c0 + w + 8, ...
#pragma unroll
  for (int rr0 = 0; rr0 < kSplitRows; rr0 += W) {
    const int rr = rr0 + warp, c = c0 + rr;
    const float* prow = th + skew_row_start(c, B) - (c + 1);   // prow[k] = theta(c, k)
    float v[B / 32];
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      v[q] = k > c ? __ldg(prow + k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      if (k >= c) tile[rr * LD + k] = -v[q];
    }
  }
  // left of the diagonal: lane = row c0 + lane, warp w takes packed rows k = w, w + 8, ...
  {
    const int c = c0 + lane;
    constexpr int U = 8;
    for (int k0 = warp; k0 < c0 + kSplitRows - 1; k0 += W * U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        v[u] = k < c ? __ldg(th + skew_row_start(k, B) + (c - k - 1)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        if (k < c) tile[lane * LD + k] = v[u];
      }
    }
  }
  __syncthreads();
  __half* qb = static_cast<__half*>(sd.Q) + (size_t)j * 512 * B;
  uint32_t* hi = reinterpret_cast<uint32_t*>(qb + (size_t)c0 * B);
  uint32_t* lo = reinterpret_cast<uint32_t*>(qb + (size_t)(B + c0) * B);
  for (int u = threadIdx.x; u < kSplitRows * B / 2; u += kUnpackThreads) {
    const int r = u / (B / 2), c2 = (u % (B / 2)) * 2;
    split_f16x2(tile[r * LD + c2], tile[r * LD + c2 + 1], hi[u], lo[u]);
  }
}

// fp32 Q at b = 256: one CTA per 128-row slab (the two slabs of a block a
// cluster), the whole chain on the tensor cores as three fp16 products per
// step, X_hi K_hi + X_hi K_lo + X_lo K_hi (fp32 accumulation; the dropped
// X_lo K_lo term is below 2^-22 of the product).  Tensor memory holds the
// slab's accumulator (128 x 256 fp32, columns [0, 256)) and X_i as the A
// operand, hi at [256, 384) and lo at [384, 512) (two fp16 per column), so
// one CTA owns an SM's tensor memory.  Warp 0 streams Kop's hi and lo parts
// (the B operand: Kop[c][k] = K[k][c], K-major) through a ring of 64-column
// chunks by TMA, every step (K does not fit in shared memory twice); warp 1
// issues the products, the 2K term among them as 2I . K over the slab's own
// K range (2I, 128 x 128 fp16, sits in shared memory beside the ring; 2 * fp16
// is exact); warps 2..9 turn the accumulator into the next X, split into its
// fp16 parts, or, after the last step, into Q = I + X_{n+1}, staged in the
// then idle ring and written
// by tensor stores once both slabs of the block are past their last read of
// Kop (cluster barrier): Q overwrites the buffer Kop lives in.
constexpr int kF32Threads = 320;
constexpr int kF32Workers = 256;
constexpr int kF32Stages = 3;
constexpr int kF32Chunk = 256 * 64 * 2;            // one part of a 64-column chunk of Kop
constexpr int kF32Stage = 2 * kF32Chunk;           // hi + lo
constexpr int kF32TwoI = 128 * 128 * 2;            // 2I over the slab's K range, fp16
constexpr int kF32Smem = 1024 + kF32Stages * kF32Stage + kF32TwoI + 256;

__global__ void __launch_bounds__(kF32Threads, 1)
    cnp_fwd_f32_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tk1,
                       const __grid_constant__ CUtensorMap tq0, const __grid_constant__ CUtensorMap tq1,
                       FwdSide f0, FwdSide f1, int n, int* err) {
  constexpr int B = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* two_i = smem + kF32Stages * kF32Stage;    // [2 k-chunks][128 rows][64 k] fp16, K-major
  uint64_t* full = reinterpret_cast<uint64_t*>(two_i + kF32TwoI);
  uint64_t* empty = full + kF32Stages;
  uint64_t* acc_full = empty + kF32Stages;
  uint64_t* x_ready = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(x_ready + 1);
  int* failed = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool second = (int)blockIdx.y >= f0.nb;
  const int j = second ? (int)blockIdx.y - f0.nb : (int)blockIdx.y;
  const CUtensorMap* tk = second ? &tk1 : &tk0;
  const CUtensorMap* tq = second ? &tq1 : &tq0;
  const int r0 = blockIdx.x * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF32Stages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(x_ready, kF32Workers);
    *failed = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  // 2I: 2.0 (fp16 0x4000) at (r, r) of the slab's K range, zero elsewhere
  for (int o = threadIdx.x * 16; o < kF32TwoI; o += kF32Threads * 16)
    *reinterpret_cast<uint4*>(two_i + o) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    *reinterpret_cast<uint16_t*>(two_i + sw128_offset(r, r, 128)) = 0x4000;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t x_hi = tmem + 256, x_lo = tmem + 384;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ Kop chunks by TMA
    if (lane == 0) {
      int it = 0, issued = 0;
      for (int i = 1; i <= n && ok; ++i)
        for (int c = 0; c < B / 64 && ok; ++c, ++it) {
          const int slot = it % kF32Stages;
          if (it >= kF32Stages &&
              !(ok = mbar_wait(empty + slot, (uint32_t)(it / kF32Stages - 1) & 1, err)))
            break;
          uint8_t* dst = ring + slot * kF32Stage;
          mbar_arrive_expect_tx(full + slot, (uint32_t)kF32Stage);
          tma_load_2d(dst, tk, 64 * c, j * 512, full + slot);
          tma_load_2d(dst + kF32Chunk, tk, 64 * c, j * 512 + 256, full + slot);
          ++issued;
        }
      if (!ok) {
        *failed = 1;
        // the copies in flight land before the CTA's memory goes (bounded)
        for (int k = (issued > kF32Stages ? issued - kF32Stages : 0); k < issued; ++k)
          mbar_wait_bounded(full + k % kF32Stages, (uint32_t)(k / kF32Stages) & 1, 1u << 16,
                            nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ products
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, B, false, false);
      // the first step's A is X_1 = K = -Kop: the slab's own rows of each
      // chunk of Kop, read with the instruction's negate-A bit (bit 13)
      const uint32_t idesc_neg = idesc | (1u << 13);
      int it = 0;
      bool pending = false;
      for (int i = 1; i <= n && ok; ++i) {
        if (!(ok = mbar_wait(x_ready, (uint32_t)(i - 1) & 1, err))) break;
        tc_fence_after();
        for (int c = 0; c < B / 64; ++c, ++it) {
          const int slot = it % kF32Stages;
          if (!(ok = mbar_wait(full + slot, (uint32_t)(it / kF32Stages) & 1, err))) break;
          tc_fence_after();
          const uint32_t bh = smem_u32(ring + slot * kF32Stage), bl = bh + kF32Chunk;
          // the chunk lies in the slab's own K range: it also carries 2I . K
          const int ci = c - 2 * (int)blockIdx.x;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t xa = (uint32_t)(32 * c + 8 * kk);   // (64 c + 16 kk) / 2
            if (i == 1) {
              const uint64_t ah = sw128_desc(bh + r0 * 128 + kk * 32, 16, 1024);
              const uint64_t al = sw128_desc(bl + r0 * 128 + kk * 32, 16, 1024);
              mma_bf16(tmem, ah, sw128_desc(bh + kk * 32, 16, 1024), idesc_neg, (c | kk) != 0);
              mma_bf16(tmem, ah, sw128_desc(bl + kk * 32, 16, 1024), idesc_neg, 1);
              mma_bf16(tmem, al, sw128_desc(bh + kk * 32, 16, 1024), idesc_neg, 1);
            } else {
              mma_bf16_ts(tmem, x_hi + xa, sw128_desc(bh + kk * 32, 16, 1024), idesc, (c | kk) != 0);
              mma_bf16_ts(tmem, x_hi + xa, sw128_desc(bl + kk * 32, 16, 1024), idesc, 1);
              mma_bf16_ts(tmem, x_lo + xa, sw128_desc(bh + kk * 32, 16, 1024), idesc, 1);
            }
            if (ci == 0 || ci == 1) {
              const uint64_t ad = sw128_desc(smem_u32(two_i) + ci * (128 * 128) + kk * 32, 16, 1024);
              mma_bf16(tmem, ad, sw128_desc(bh + kk * 32, 16, 1024), idesc, 1);
              mma_bf16(tmem, ad, sw128_desc(bl + kk * 32, 16, 1024), idesc, 1);
            }
          }
          mma_commit(empty + slot);
          pending = true;
        }
        if (!ok) break;
        mma_commit(acc_full);
      }
      if (!ok) {
        *failed = 1;
        // the products issued complete before tensor memory is freed (bounded)
        if (pending && it > 0)
          mbar_wait_bounded(empty + (it - 1) % kF32Stages, (uint32_t)((it - 1) / kF32Stages) & 1,
                            1u << 16, nullptr);
      }
    }
  } else {
    // ------------------------------------------------ conversions
    const int quarter = warp % 4, half = (warp - 2) / 4;
    const int r = quarter * 32 + lane, row = r0 + r;   // TMEM lane, row of the block
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // X_1 needs no conversion (the first products read it from the ring)
    mbar_arrive(x_ready);
    for (int i = 1; i <= n && ok; ++i) {
      if (!(ok = mbar_wait(acc_full, (uint32_t)(i - 1) & 1, err))) break;
      tc_fence_after();
      for (int c0 = half * 128; c0 < half * 128 + 128; c0 += 32) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_off + (uint32_t)c0, acc);
        tmem_ld_wait();
        tmem_regs_ready(acc);
        float x[32];   // X_{i+1}: the products hold the 2K term
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(acc[e]);
        if (i < n) {
          uint32_t h[16], l[16];
          float big = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            split_f16x2(x[2 * e], x[2 * e + 1], h[e], l[e]);
            big = fmaxf(big, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
          }
          if (big >= 65504.f) raise_device_error(err, POETX_ERR_RANGE);   // beyond fp16
          tmem_st16(x_hi + lane_off + (uint32_t)(c0 / 2), h);
          tmem_st16(x_lo + lane_off + (uint32_t)(c0 / 2), l);
        } else {
          // Q = I + X_{n+1} into the idle ring: 128 x 32 fp32 boxes (128-byte
          // swizzle: row r's 16-byte chunk q at r * 128 + (q ^ (r % 8)) * 16)
          if (__any_sync(0xffffffffu, (unsigned)(row - c0) < 32u)) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (row == c0 + e) x[e] += 1.f;
          }
          uint8_t* box = ring + (c0 / 32) * (128 * 128) + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(box + ((q ^ (r & 7)) << 4)) =
                make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
      }
      if (i < n) {
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(x_ready);
      }
    }
    if (!ok) *failed = 1;
    fence_proxy_async_smem();   // the staged Q, for the tensor stores
  }
  tc_fence_before();
  __syncthreads();
  // both slabs of the block are past their last read of Kop (the ring's
  // copies, the 2K rows): Q may overwrite it
  cluster_sync();
  if (threadIdx.x == 0 && *failed == 0) {
    for (int q = 0; q < B / 32; ++q) tma_store_2d(tq, ring + q * (128 * 128), 32 * q, j * B + r0);
    bulk_commit();
    bulk_wait0();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ====================================================================== backward
struct Side {
  const float* theta;
  const float* dQ;     // dQ as n_part partial-sum slots [n_part][nb, b, b]; summed in slot order
  int n_part;
  __nv_bfloat16* Kd;   // K, [nb, b, b] bf16: the B operand of X -> X K^T
  __nv_bfloat16* Td;   // K^T = -K, [nb, b, b] bf16: the first A operand X_1
  __nv_bfloat16* Gd;   // dQ in bf16, [nb, b, b]
  float* dK;           // dK of every block, fp32 [nb, b, b] (read back when packing)
  float* dtheta;
  int nb;
};

constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 32;

// Kd[j] = bf16(K_j), Td[j] = -Kd[j], Gd[j] = bf16(dQ_j) for both sides; CTA
// (x, y, z) takes the 32-row group x of block y: the z-th quarter of the
// group's dQ columns (the partial-sum slots added in order), and for z = 0
// also the group's rows of K, assembled in shared memory (row pitch B + 2
// halves, so the column writes fall in distinct banks): entries right of the
// diagonal come from the packed rows of the group, the ones left of it from
// the packed rows above, which hold the group's columns contiguously.  All
// loads are issued before their stores.
constexpr int kPrepZ = 4;
// parts of the CNP backward (cnp_bwd_side): the dense K and K^T from theta,
// the summed dQ as bf16 G, the chain
constexpr int kPrepK = 1, kPrepG = 2, kChain = 4;

template <int B>
__global__ void __launch_bounds__(kPrepThreads)
    cnp_prep_kernel(Side s0, Side s1, int what) {
  __shared__ __nv_bfloat16 tile[kPrepRows * (B + 2)];
  constexpr int LD = B + 2;
  constexpr int P = B * (B - 1) / 2;
  const bool second = (int)blockIdx.y >= s0.nb;
  const Side& sd = second ? s1 : s0;
  const int j = second ? (int)blockIdx.y - s0.nb : (int)blockIdx.y;
  const int c0 = blockIdx.x * kPrepRows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // ---- dQ: rows [c0, c0 + 32), columns of quarter z -> bf16
  if (what & kPrepG) {
    constexpr int QC = B / kPrepZ;   // columns of the quarter
    const float4* g4 = reinterpret_cast<const float4*>(sd.dQ + ((size_t)j * B + c0) * B);
    const size_t slot4 = (size_t)sd.nb * B * B / 4;
    uint4* gd = reinterpret_cast<uint4*>(sd.Gd + ((size_t)j * B + c0) * B);
    for (int u = threadIdx.x; u < kPrepRows * QC / 8; u += kPrepThreads) {
      const int e8 = ((u / (QC / 8)) * B + (int)blockIdx.z * QC + (u % (QC / 8)) * 8) / 8;
      // slots added in order 0, 1, ...; up to 8 slots' loads in flight at a time
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
      for (int p0 = 0; p0 < sd.n_part; p0 += 8) {
        float4 va[8], vc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (p0 + q < sd.n_part) {
            va[q] = __ldg(g4 + (p0 + q) * slot4 + 2 * e8);
            vc[q] = __ldg(g4 + (p0 + q) * slot4 + 2 * e8 + 1);
          }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (p0 + q < sd.n_part) {
            a.x += va[q].x; a.y += va[q].y; a.z += va[q].z; a.w += va[q].w;
            c.x += vc[q].x; c.y += vc[q].y; c.z += vc[q].z; c.w += vc[q].w;
          }
      }
      gd[e8] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(c.x, c.y),
                          pack_bf16x2(c.z, c.w));
    }
  }
  if (blockIdx.z != 0 || !(what & kPrepK)) return;
  // ---- K and K^T rows of the group
  const float* th = sd.theta + (size_t)j * P;
  constexpr int W = kPrepThreads / 32;
#pragma unroll
  for (int rr0 = 0; rr0 < kPrepRows; rr0 += W) {
    const int rr = rr0 + warp, c = c0 + rr;
    const float* prow = th + skew_row_start(c, B) - (c + 1);   // prow[k] = theta(c, k)
    float v[B / 32];
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      v[q] = k > c ? __ldg(prow + k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < B / 32; ++q) {
      const int k = q * 32 + lane;
      if (k >= c) tile[rr * LD + k] = __float2bfloat16_rn(v[q]);
    }
  }
  {
    const int c = c0 + lane;
    constexpr int U = 8;
    for (int k0 = warp; k0 < c0 + kPrepRows - 1; k0 += W * U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        v[u] = k < c ? __ldg(th + skew_row_start(k, B) + (c - k - 1)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = k0 + u * W;
        if (k < c) tile[lane * LD + k] = __float2bfloat16_rn(-v[u]);
      }
    }
  }
  __syncthreads();
  uint32_t* kd = reinterpret_cast<uint32_t*>(sd.Kd + ((size_t)j * B + c0) * B);
  uint32_t* td = reinterpret_cast<uint32_t*>(sd.Td + ((size_t)j * B + c0) * B);
  for (int u = threadIdx.x; u < kPrepRows * B / 2; u += kPrepThreads) {
    const int r = u / (B / 2), c2 = (u % (B / 2)) * 2;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + r * LD + c2);
    kd[u] = w;
    td[u] = w ^ 0x80008000u;
  }
}

// One cluster per block: CTA (row half mh, column slab ns) of the cluster
// (rank = ns * MH + mh; MH = B / 128 row halves, NS = B / 64 slabs of 64
// columns) runs the transpose of the adjoint chain on rows [128 mh, 128 mh +
// 128) and columns [64 ns, 64 ns + 64) of
//   X^T_1 = K, Y^T_1 = G^T,
//   X^T_{i+1} = K X^T_i + 2K,  Y^T_{i+1} = G^T X^T_i + K Y^T_i + 2G^T,  dK^T = Y^T_{n+1}
// (the transpose of X_{i+1} = X_i A + 2A, Y_{i+1} = X_i G + Y_i A + 2G with
// A = K^T).  The A operands are resident for the whole chain: the CTA's rows
// of K (K-major) and of G^T (MN-major: rows of G); the B operands are the
// slab's columns of X^T_i and Y^T_i over all B rows.  Each step's MMAs
// (M = 128, N = 64, K = 16, fp32 in TMEM) give the CTA's rows of the next B
// operands: the workers write them as bf16 into the CTA's own B buffers and
// one bulk copy per operand sends the same rows into the other row half's
// buffers (the only exchange; both halves' MMAs of a step signal both CTAs
// through one multicast commit, so a buffer is overwritten only after every
// MMA reading it has finished).  The terms 2K and 2G^T enter as MMAs of the
// slab's 64 columns of K and G^T against a 2I tile.  At the end the workers
// write the CTA's tile of dK^T (fp32) to the workspace, and after a cluster
// barrier the cluster packs dtheta(i, k) = dK[i][k] - dK[k][i] = dK^T[k][i] -
// dK^T[i][k] (i < k) from 32 x 32 tile pairs, every entry written once.
constexpr int kBwdThreads = 192;   // warp 0: TMA and copies; warp 1: TMEM + MMA; warps 2..5: workers
constexpr int kBwdWorkers = 128;
constexpr int kPackPitch = 33;     // fp32 pitch of the 32 x 32 transpose tiles

template <int B>
struct BwdGeo {
  static constexpr int MH = B / 128, NS = B / 64, CL = MH * NS;
  static constexpr int a_bytes = 128 * B * 2;   // one A operand: 128 rows x B
  static constexpr int b_bytes = B * 128;       // one B operand: B rows x 64 columns
  static constexpr int i_bytes = 64 * 128;      // the 2I tile
  static constexpr int half_bytes = 128 * 128;  // a row half of a B operand (MH = 2)
  static_assert(MH == 1 || half_bytes * MH == b_bytes, "the row halves tile a B operand");
  static constexpr int off_a1 = 1024;
  static constexpr int off_a2 = off_a1 + a_bytes;
  static constexpr int off_bx = off_a2 + a_bytes;
  static constexpr int off_by = off_bx + b_bytes;
  static constexpr int off_bi = off_by + b_bytes;
  static constexpr int smem = 1024 + off_bi + i_bytes;   // + alignment slack
  static constexpr uint32_t load_bytes = 2 * a_bytes + 2 * b_bytes;
};

template <int B>
__global__ void __launch_bounds__(kBwdThreads, 1)
    cnp_bwd_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tg0,
                   const __grid_constant__ CUtensorMap tk1, const __grid_constant__ CUtensorMap tg1,
                   Side s0, Side s1, int n, int* err) {
  using Geo = BwdGeo<B>;
  constexpr int MH = Geo::MH, CL = Geo::CL;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int blk = (int)blockIdx.x / CL;
  const bool second = blk >= s0.nb;
  const Side& sd = second ? s1 : s0;
  const CUtensorMap* tk = second ? &tk1 : &tk0;
  const CUtensorMap* tg = second ? &tg1 : &tg0;
  const int j = second ? blk - s0.nb : blk;
  const int rank = (int)cluster_ctarank();
  const int mh = rank % MH, ns = rank / MH;
  const int peer = rank ^ 1;   // the other row half of the slab (MH == 2)
  uint8_t* a1 = smem + Geo::off_a1;
  uint8_t* a2 = smem + Geo::off_a2;
  uint8_t* bx = smem + Geo::off_bx;
  uint8_t* by = smem + Geo::off_by;
  uint8_t* bi = smem + Geo::off_bi;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* ops_full = bars;        // operands loaded and the 2I tile written
  uint64_t* mma_done = bars + 1;    // this step's MMAs of both row halves have completed
  uint64_t* rows_ready = bars + 2;  // the workers have written this CTA's rows of the next B operands
  uint64_t* recv = bars + 3;        // the other row half's rows have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(ops_full, 2);
    mbar_init(mma_done, MH);
    mbar_init(rows_ready, kBwdWorkers);
    mbar_init(recv, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // every CTA's barriers are initialised before any remote arrival or copy
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t dx = tmem_base, dy = tmem_base + 64;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ TMA: the operands; then the row exchange
    if (lane == 0) {
      mbar_arrive_expect_tx(ops_full, Geo::load_bytes);
      const int r0 = j * B;
      for (int q = 0; q < B / 64; ++q)       // A1: K rows [128 mh, +128), K-major
        for (int rb = 0; rb < 2; ++rb)
          tma_load_2d(a1 + q * (128 * 128) + rb * (64 * 128), tk, q * 64, r0 + 128 * mh + 64 * rb, ops_full);
      for (int mc = 0; mc < 2; ++mc)         // A2: G^T rows = G columns [128 mh, +128), MN-major
        for (int kb = 0; kb < B / 64; ++kb)
          tma_load_2d(a2 + mc * Geo::b_bytes + kb * (64 * 128), tg, 128 * mh + 64 * mc, r0 + 64 * kb, ops_full);
      for (int kb = 0; kb < B / 64; ++kb)    // B_X = X^T_1 = K columns of the slab, MN-major
        tma_load_2d(bx + kb * (64 * 128), tk, 64 * ns, r0 + 64 * kb, ops_full);
      for (int q = 0; q < B / 64; ++q)       // B_Y = Y^T_1 = G^T: rows of G in the slab, K-major
        tma_load_2d(by + q * (64 * 128), tg, q * 64, r0 + 64 * ns, ops_full);
      if constexpr (MH == 2) {
        // after each step but the last: this CTA's new rows to the other half
        const uint32_t rx = mapa_shared(smem_u32(bx + mh * Geo::half_bytes), (uint32_t)peer);
        const uint32_t ry = mapa_shared(smem_u32(by + mh * Geo::half_bytes), (uint32_t)peer);
        const uint32_t rb = mapa_shared(smem_u32(recv), (uint32_t)peer);
        for (int i = 1; i < n && ok; ++i) {
          if (!(ok = mbar_wait(rows_ready, (i - 1) & 1, err))) break;
          bulk_copy_s2cluster(rx, bx + mh * Geo::half_bytes, Geo::half_bytes, rb);
          bulk_copy_s2cluster(ry, by + mh * Geo::half_bytes, Geo::half_bytes, rb);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t id_km = idesc_bf16(128, 64, false, true);    // A K-major, B MN-major
      const uint32_t id_kk = idesc_bf16(128, 64, false, false);   // A K-major, B K-major
      const uint32_t id_mm = idesc_bf16(128, 64, true, true);     // A MN-major, B MN-major
      const uint32_t id_mk = idesc_bf16(128, 64, true, false);    // A MN-major, B K-major
      const uint32_t a1b = smem_u32(a1), a2b = smem_u32(a2), bxb = smem_u32(bx), byb = smem_u32(by),
                     bib = smem_u32(bi);
      const uint16_t mask = (uint16_t)((1u << rank) | (1u << peer));
      ok = mbar_wait(ops_full, 0, err);
      for (int i = 1; i <= n && ok; ++i) {
        if (i > 1) {
          if (!(ok = mbar_wait(rows_ready, (i - 2) & 1, err))) break;
          if constexpr (MH == 2)
            if (!(ok = mbar_wait(recv, (i - 2) & 1, err))) break;
        }
        tc_fence_after();
        // X^T_{i+1} = K X^T_i + 2K (not needed after the last step)
        if (i < n) {
#pragma unroll 4
          for (int kk = 0; kk < B / 16; ++kk)
            mma_bf16(dx, sw128_desc(a1b + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024),
                     sw128_desc(bxb + kk * 2048, Geo::b_bytes, 1024), id_km, kk != 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(dx, sw128_desc(a1b + ns * (128 * 128) + kk * 32, 16, 1024),
                     sw128_desc(bib + kk * 32, 16, 1024), id_kk, 1);
        }
        // Y^T_{i+1} = G^T X^T_i + K Y^T_i + 2G^T
#pragma unroll 4
        for (int kk = 0; kk < B / 16; ++kk)
          mma_bf16(dy, sw128_desc(a2b + kk * 2048, Geo::b_bytes, 1024),
                   sw128_desc(bxb + kk * 2048, Geo::b_bytes, 1024), id_mm, kk != 0);
        if (i == 1) {   // Y^T_1 = G^T as loaded: K-major
#pragma unroll 4
          for (int kk = 0; kk < B / 16; ++kk)
            mma_bf16(dy, sw128_desc(a1b + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024),
                     sw128_desc(byb + (kk >> 2) * (64 * 128) + (kk & 3) * 32, 16, 1024), id_kk, 1);
        } else {
#pragma unroll 4
          for (int kk = 0; kk < B / 16; ++kk)
            mma_bf16(dy, sw128_desc(a1b + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024),
                     sw128_desc(byb + kk * 2048, Geo::b_bytes, 1024), id_km, 1);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(dy, sw128_desc(a2b + (4 * ns + kk) * 2048, Geo::b_bytes, 1024),
                   sw128_desc(bib + kk * 32, 16, 1024), id_mk, 1);
        // the other half's rows of the next operands land on `recv`; expected
        // before this step's commit, so before the other half may send them
        if constexpr (MH == 2)
          if (i < n) mbar_arrive_expect_tx(recv, 2 * Geo::half_bytes);
        if constexpr (MH == 2) mma_commit_multicast(mma_done, mask);
        else mma_commit(mma_done);
      }
    }
  } else {
    // ------------------------------------------------ workers: 2I tile, next operands, dK^T
    const int wt = threadIdx.x - 64;
    const int quarter = warp % 4;
    const int m = quarter * 32 + lane;   // TMEM lane = row of the CTA's half
    const int k = 128 * mh + m;          // its row in the B operands
    for (int u = wt; u < Geo::i_bytes / 16; u += kBwdWorkers)
      reinterpret_cast<uint4*>(bi)[u] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("bar.sync 1, %0;" ::"n"(kBwdWorkers) : "memory");
    if (wt < 64)   // 2.0 at (r, r): K-major [64 n][64 k]
      *reinterpret_cast<__nv_bfloat16*>(bi + sw128_offset(wt, wt, 64)) = __float2bfloat16_rn(2.f);
    fence_proxy_async_smem();
    asm volatile("bar.sync 1, %0;" ::"n"(kBwdWorkers) : "memory");
    if (wt == 0) mbar_arrive(ops_full);
    for (int i = 1; i <= n && ok; ++i) {
      if (!(ok = mbar_wait(mma_done, (i - 1) & 1, err))) break;
      tc_fence_after();
      const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
      if (i < n) {
        // row k of X^T_{i+1} and Y^T_{i+1}: 64 columns each, bf16, MN-major (128-byte swizzle)
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t r[2][32];
          const uint32_t col = t == 0 ? dx : dy;
          tmem_ld32(col + lrow, r[0]);
          tmem_ld32(col + 32u + lrow, r[1]);
          tmem_ld_wait();
          tmem_regs_ready(r[0]);
          tmem_regs_ready(r[1]);
          uint8_t* row = (t == 0 ? bx : by) + k * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[c >> 2][(c & 3) * 8 + e]);
            *reinterpret_cast<uint4*>(row + ((c ^ (k & 7)) << 4)) = pack8(v);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(rows_ready);
      } else {
        // dK^T rows: [128 mh + m][64 ns, +64) of block j, fp32
        uint32_t r[2][32];
        tmem_ld32(dy + lrow, r[0]);
        tmem_ld32(dy + 32u + lrow, r[1]);
        tmem_ld_wait();
        tmem_regs_ready(r[0]);
        tmem_regs_ready(r[1]);
        float4* dst = reinterpret_cast<float4*>(sd.dK + ((size_t)j * B + k) * B + 64 * ns);
#pragma unroll
        for (int q = 0; q < 16; ++q)
          dst[q] = make_float4(__uint_as_float(r[q >> 3][(q & 7) * 4]), __uint_as_float(r[q >> 3][(q & 7) * 4 + 1]),
                               __uint_as_float(r[q >> 3][(q & 7) * 4 + 2]),
                               __uint_as_float(r[q >> 3][(q & 7) * 4 + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // every CTA's dK^T tile is written (release/acquire at cluster scope), no
  // copy into or commit onto another CTA is outstanding
  cluster_sync();
  // ---- pack: 32 x 32 tile pairs (ti <= tk) shared round-robin by the cluster's CTAs and warps
  {
    constexpr int NT = B / 32;
    constexpr int W = kBwdThreads / 32;
    float* tA = reinterpret_cast<float*>(smem + Geo::off_a1) + warp * (2 * 32 * kPackPitch);
    float* tB = tA + 32 * kPackPitch;
    const float* dKt = sd.dK + (size_t)j * B * B;
    float* dth = sd.dtheta + (size_t)j * (B * (B - 1) / 2);
    int t = 0;
    for (int ti = 0; ti < NT; ++ti)
      for (int tk = ti; tk < NT; ++tk, ++t) {
        if (t % CL != rank || (t / CL) % W != warp) continue;
        // tA[ii][kk] = dK^T[32ti+ii][32tk+kk],  tB[kk][ii] = dK^T[32tk+kk][32ti+ii]: all 64
        // row segments requested before any is stored (other CTAs' rows: read at L2)
        float va[32], vb[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          va[ii] = __ldcg(dKt + (size_t)(32 * ti + ii) * B + 32 * tk + lane);
          vb[ii] = __ldcg(dKt + (size_t)(32 * tk + ii) * B + 32 * ti + lane);
        }
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          tA[ii * kPackPitch + lane] = va[ii];
          tB[ii * kPackPitch + lane] = vb[ii];
        }
        __syncwarp();
        for (int ii = 0; ii < 32; ++ii) {
          const int i = 32 * ti + ii, kc = 32 * tk + lane;
          if (i < kc)   // dK[i][kc] - dK[kc][i] = dK^T[kc][i] - dK^T[i][kc]
            dth[skew_row_start(i, B) + (kc - i - 1)] = tB[lane * kPackPitch + ii] - tA[ii * kPackPitch + lane];
        }
        __syncwarp();
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 128);
  }
}

constexpr int kRingThreads = 320;   // warp 0: TMEM + MMA; warp 1: TMA; warps 2..9: workers
constexpr int kRingWorkers = 256;

// The narrow form of the same chain, for running beside a kernel that holds
// most SMs (the R side's chain beside the g_u GEMM): two CTAs per block.
// One CTA = one 128-row slab of one block; for B = 256 the two slabs of a
// block form a cluster.  With A = K^T and G = dL/dQ the chain
//   X_1 = A, Y_1 = G,  X_{i+1} = X_i A + 2A,  Y_{i+1} = X_i G + Y_i A + 2G,  dK = Y_{n+1}
// runs as tcgen05.mma into TMEM.  X_1 and Y_1 arrive by TMA (prepared K^T and
// G rows); the B operands K (for X A, Y A) and G^T stream through a TMA ring;
// the terms 2A and 2G enter as extra MMAs whose A operand is 2I on the
// slab's own rows (only the two 64-wide K chunks of the slab are non-zero), so
// between steps the workers only convert TMEM to bf16 operands.  dK goes to
// the workspace; after a cluster barrier both slabs pack
//   dtheta(i,k) = dK[i][k] - dK[k][i]  (i < k)
// from 32 x 32 tile pairs transposed through shared memory, each CTA taking
// half of the tiles, every packed entry written exactly once.
template <int B>
__global__ void __launch_bounds__(kRingThreads, 1)
    cnp_bwd_ring_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tg0,
                   const __grid_constant__ CUtensorMap tt0, const __grid_constant__ CUtensorMap tk1,
                   const __grid_constant__ CUtensorMap tg1, const __grid_constant__ CUtensorMap tt1,
                   Side s0, Side s1, int n, int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const bool second = (int)blockIdx.y >= s0.nb;
  const Side& sd = second ? s1 : s0;
  const CUtensorMap* tk = second ? &tk1 : &tk0;
  const CUtensorMap* tg = second ? &tg1 : &tg0;
  const CUtensorMap* tt = second ? &tt1 : &tt0;
  const int j = second ? (int)blockIdx.y - s0.nb : (int)blockIdx.y;
  const int slab = blockIdx.x;
  const int r0 = slab * 128;
  constexpr int a_bytes = 128 * B * 2;
  constexpr int i_bytes = 128 * 128 * 2;
  constexpr int chunk_bytes = B * 64 * 2;
  constexpr int kchunks = B / 64;
  constexpr uint32_t ncols = 2 * B;
  uint8_t* ax = smem;
  uint8_t* ay = smem + a_bytes;
  uint8_t* itl = smem + 2 * a_bytes;   // 2I on the slab's K range, [128 rows][128 k], K-major
  uint8_t* ring = itl + i_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + stages * chunk_bytes);
  uint64_t* bfull = bars;
  uint64_t* bempty = bfull + kMaxStages;
  uint64_t* afull = bempty + kMaxStages;
  uint64_t* stepdone = afull + 1;
  uint64_t* a0full = stepdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(a0full + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kMaxStages; ++st) {
      mbar_init(bfull + st, 1);
      mbar_init(bempty + st, 1);
    }
    mbar_init(afull, kRingWorkers);
    mbar_init(stepdone, 1);
    mbar_init(a0full, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool ok = true;

  if (warp == 1) {
    // ------------------------------------------------ TMA: X_1, Y_1, then per step K chunks and G^T chunks
    if (lane == 0) {
      mbar_arrive_expect_tx(a0full, (uint32_t)(2 * a_bytes));
      for (int q = 0; q < kchunks; ++q) {
        tma_load_2d(ax + q * (128 * 128), tt, q * 64, j * B + r0, a0full);   // K^T rows
        for (int h = 0; h < 2; ++h)                                         // G rows
          tma_load_2d(ay + q * (128 * 128) + h * (64 * 128), tg, q * 64, j * B + r0 + 64 * h, a0full);
      }
      int st = 0;
      uint32_t ph = 0;
      for (int i = 1; i <= n && ok; ++i)
        for (int c = 0; c < 2 * kchunks && ok; ++c) {
          if (!(ok = mbar_wait(bempty + st, ph ^ 1, err))) break;
          mbar_arrive_expect_tx(bfull + st, (uint32_t)(B * 128));
          uint8_t* dst = ring + st * chunk_bytes;
          if (c < kchunks) {
            tma_load_2d(dst, tk, c * 64, j * B, bfull + st);           // B[cc][k] = K[cc][k]
          } else {
            const int kc = c - kchunks;
            for (int q = 0; q < B / 64; ++q)                          // B[cc][k] = G[k][cc]
              tma_load_2d(dst + q * 8192, tg, q * 64, j * B + kc * 64, bfull + st);
          }
          if (++st == stages) { st = 0; ph ^= 1; }
        }
    }
  } else if (warp == 0) {
    // ------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t idk = idesc_bf16(128, B, false, false);
      const uint32_t idg = idesc_bf16(128, B, false, true);
      const uint32_t dx = tmem_base, dy = tmem_base + (uint32_t)B;
      const uint32_t axb = smem_u32(ax), ayb = smem_u32(ay), itb = smem_u32(itl);
      int st = 0;
      uint32_t ph = 0;
      ok = mbar_wait(a0full, 0, err);
      for (int i = 1; i <= n && ok; ++i) {
        if (!(ok = mbar_wait(afull, (i - 1) & 1, err))) break;
        tc_fence_after();
        for (int c = 0; c < 2 * kchunks && ok; ++c) {
          if (!(ok = mbar_wait(bfull + st, ph, err))) break;
          tc_fence_after();
          const uint32_t bb = smem_u32(ring + st * chunk_bytes);
          const int kc = c % kchunks;
          const int ic = kc - r0 / 64;                 // chunk of the 2I tile, when 0 or 1
          const bool in_slab = ic == 0 || ic == 1;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t xdesc = sw128_desc(axb + kc * 128 * 128 + kk * 32, 16, 1024);
            const uint64_t idsc = sw128_desc(itb + (in_slab ? ic : 0) * 128 * 128 + kk * 32, 16, 1024);
            if (c < kchunks) {
              const uint64_t bdesc = sw128_desc(bb + kk * 32, 16, 1024);
              const uint32_t acc = (kc | kk) != 0;
              if (i < n) mma_bf16(dx, xdesc, bdesc, idk, acc);                    // X A
              mma_bf16(dy, sw128_desc(ayb + kc * 128 * 128 + kk * 32, 16, 1024), bdesc, idk,
                       acc);                                                    // Y A
              if (i < n && in_slab) mma_bf16(dx, idsc, bdesc, idk, 1);          // + 2A
            } else {
              const uint64_t bdesc = sw128_desc(bb + kk * 2048, 8192, 1024);
              mma_bf16(dy, xdesc, bdesc, idg, 1);                              // X G
              if (in_slab) mma_bf16(dy, idsc, bdesc, idg, 1);                   // + 2G
            }
          }
          mma_commit(bempty + st);
          if (++st == stages) { st = 0; ph ^= 1; }
        }
        mma_commit(stepdone);
      }
    }
  } else {
    // ------------------------------------------------ workers: 2I tile, operands, dK rows
    const int wt = threadIdx.x - 64;
    const int quarter = warp % 4;
    const int half = (warp - 2) / 4;
    const int r = quarter * 32 + lane;
    for (int u = wt; u < i_bytes / 16; u += kRingWorkers)
      reinterpret_cast<uint4*>(itl)[u] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("bar.sync 1, %0;" ::"n"(kRingWorkers) : "memory");
    if (wt < 128)   // 2.0 at (r, r) of the slab's K range
      *reinterpret_cast<__nv_bfloat16*>(itl + sw128_offset(wt, wt, 128)) = __float2bfloat16_rn(2.f);
    fence_proxy_async_smem();
    mbar_arrive(afull);
    for (int i = 2; i <= n && ok; ++i) {
      if (!(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
      tc_fence_after();
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t rx[32], ry[32];
        tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rx);
        tmem_ld32(tmem_base + (uint32_t)(B + c0) + ((uint32_t)(quarter * 32) << 16), ry);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float x[8], y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = __uint_as_float(rx[8 * g + e]);
            y[e] = __uint_as_float(ry[8 * g + e]);
          }
          *reinterpret_cast<uint4*>(ax + sw128_offset(r, c0 + 8 * g, 128)) = pack8(x);
          *reinterpret_cast<uint4*>(ay + sw128_offset(r, c0 + 8 * g, 128)) = pack8(y);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(afull);
    }
    // dK = Y_{n+1}: the slab's rows to the workspace, 32 x 32 tiles turned
    // through the warp's own shared-memory tile (the chain's operand buffers
    // are free once the last step is done) so that each store is a full row
    // segment of 128 bytes
    if (ok && (ok = mbar_wait(stepdone, (n - 1) & 1, err))) {
      tc_fence_after();
      float* tt = reinterpret_cast<float*>(smem) + warp * (2 * 32 * kPackPitch);
      float* dtile = sd.dK + ((size_t)j * B + r0 + quarter * 32) * B;
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t ry[32];
        tmem_ld32(tmem_base + (uint32_t)(B + c0) + ((uint32_t)(quarter * 32) << 16), ry);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) tt[lane * kPackPitch + e] = __uint_as_float(ry[e]);
        __syncwarp();
#pragma unroll 8
        for (int rr = 0; rr < 32; ++rr) dtile[(size_t)rr * B + c0 + lane] = tt[rr * kPackPitch + lane];
        __syncwarp();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // every slab's dK rows are written (release/acquire at cluster scope)
  if constexpr (B == 256) cluster_sync();
  // ---- pack: 32 x 32 tile pairs (ti <= tk) shared round-robin by the CTAs and warps
  {
    constexpr int NT = B / 32;
    constexpr int CT = B / 128;   // CTAs of the block
    float* tA = reinterpret_cast<float*>(smem) + warp * (2 * 32 * kPackPitch);
    float* tB = tA + 32 * kPackPitch;
    const float* dKj = sd.dK + (size_t)j * B * B;
    float* dth = sd.dtheta + (size_t)j * (B * (B - 1) / 2);
    int t = 0;
    for (int ti = 0; ti < NT; ++ti)
      for (int tk = ti; tk < NT; ++tk, ++t) {
        if (t % CT != slab || (t / CT) % (kRingThreads / 32) != warp) continue;
        // A[ii][kk] = dK[32ti+ii][32tk+kk],  Bt[kk][ii] = dK[32tk+kk][32ti+ii]: all 64
        // row segments are requested before any is stored (one round trip to L2;
        // the partner slab's rows were written by another CTA: read at L2)
        float va[32], vb[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          va[ii] = __ldcg(dKj + (size_t)(32 * ti + ii) * B + 32 * tk + lane);
          vb[ii] = __ldcg(dKj + (size_t)(32 * tk + ii) * B + 32 * ti + lane);
        }
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
          tA[ii * kPackPitch + lane] = va[ii];
          tB[ii * kPackPitch + lane] = vb[ii];
        }
        __syncwarp();
        for (int ii = 0; ii < 32; ++ii) {
          const int i = 32 * ti + ii, k = 32 * tk + lane;
          if (i < k)
            dth[skew_row_start(i, B) + (k - i - 1)] = tA[ii * kPackPitch + lane] - tB[lane * kPackPitch + ii];
        }
        __syncwarp();
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

namespace {

// fp32 Q at b = 256: the split unpack, then the chain in 2-CTA clusters.
poetx_status cnp_fwd_f32_launch(const float* theta0, int nb0, const float* theta1, int nb1, int n,
                                void* Q0, void* Q1, cudaStream_t s) {
  FwdSide f0{theta0, Q0, nb0}, f1{theta1, Q1, nb1};
  const FwdSide& t1 = nb1 > 0 ? f1 : f0;
  const FwdSide& t0 = nb0 > 0 ? f0 : f1;
  // Kop hi / lo in the Q buffers as fp16 [nb * 512][256]; Q as fp32 [nb * 256][256]
  CUtensorMap tk0, tk1, tq0, tq1;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType h16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_tmap_2d(&tk0, t0.Q, h16, 2, (uint64_t)t0.nb * 512, 256, 256, 64, sw) ||
      !make_tmap_2d(&tk1, t1.Q, h16, 2, (uint64_t)t1.nb * 512, 256, 256, 64, sw) ||
      !make_tmap_2d(&tq0, t0.Q, f32, 4, (uint64_t)t0.nb * 256, 256, 128, 32, sw) ||
      !make_tmap_2d(&tq1, t1.Q, f32, 4, (uint64_t)t1.nb * 256, 256, 128, 32, sw))
    return POETX_ERR_CUDA;
  {
    KernelScope ks_("tc_cnp_unpack_f32", s);
    cnp_unpack_split_kernel<<<dim3(256 / kSplitRows, nb0 + nb1), kUnpackThreads, 0, s>>>(f0, f1);
  }
  poetx_status st = check_launch();
  if (st != POETX_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, nb0 + nb1);
  cfg.blockDim = dim3(kF32Threads);
  cfg.dynamicSmemBytes = kF32Smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (set_max_dynamic_smem((const void*)cnp_fwd_f32_kernel, kF32Smem) != cudaSuccess)
    return check_launch();
  KernelScope ks_("tc_cnp_fwd_f32", s);
  cudaLaunchKernelEx(&cfg, cnp_fwd_f32_kernel, tk0, tk1, tq0, tq1, f0, f1, n, device_error_word());
  return check_launch();
}

}  // namespace

poetx_status cnp_fwd_pair_bf16ops(const float* theta0, int nb0, const float* theta1, int nb1,
                                  int b, int n, void* Q0, void* Q1, bool out_f32, cudaStream_t s) {
  if (nb0 + nb1 <= 0) return POETX_OK;
  if (!cnp_supported(b) || n < 1 || nb0 + nb1 > 65535) return POETX_ERR_UNSUPPORTED;
  if (out_f32)
    return b == 256 ? cnp_fwd_f32_launch(theta0, nb0, theta1, nb1, n, Q0, Q1, s)
                    : POETX_ERR_UNSUPPORTED;
  FwdSide f0{theta0, Q0, nb0}, f1{theta1, Q1, nb1};
  const FwdSide& t1 = nb1 > 0 ? f1 : f0;
  const FwdSide& t0 = nb0 > 0 ? f0 : f1;
  CUtensorMap tk0, tk1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_2d(&tk0, t0.Q, bf, 2, (uint64_t)t0.nb * b, (uint64_t)b, (uint32_t)b, 64, sw) ||
      !make_tmap_2d(&tk1, t1.Q, bf, 2, (uint64_t)t1.nb * b, (uint64_t)b, (uint32_t)b, 64, sw))
    return POETX_ERR_CUDA;
  {
    KernelScope ks_("tc_cnp_unpack", s);
    if (b == 256)
      cnp_unpack_kernel<256><<<dim3(256 / kUnpackRows, nb0 + nb1), kUnpackThreads, 0, s>>>(f0, f1);
    else
      cnp_unpack_kernel<128><<<dim3(128 / kUnpackRows, nb0 + nb1), kUnpackThreads, 0, s>>>(f0, f1);
  }
  poetx_status st = check_launch();
  if (st != POETX_OK) return st;
  const int smem = b * b * 2 + 128 * b * 2 + 1024 + 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(b / 128, nb0 + nb1);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = b / 128;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int* err = device_error_word();
  KernelScope ks_("tc_cnp_fwd", s);
  cudaError_t e;
  if (b == 256) {
    set_max_dynamic_smem((const void*)cnp_fwd_kernel<256>, smem);
    e = cudaLaunchKernelEx(&cfg, cnp_fwd_kernel<256>, tk0, tk1, f0, f1, n, err);
  } else {
    set_max_dynamic_smem((const void*)cnp_fwd_kernel<128>, smem);
    e = cudaLaunchKernelEx(&cfg, cnp_fwd_kernel<128>, tk0, tk1, f0, f1, n, err);
  }
  if (e != cudaSuccess) return check_launch();
  return check_launch();
}

poetx_status cnp_fwd_bf16ops(const float* theta, int nb, int b, int n, void* Q, bool out_f32,
                             cudaStream_t s) {
  return cnp_fwd_pair_bf16ops(theta, nb, theta, 0, b, n, Q, Q, out_f32, s);
}

size_t cnp_bwd_workspace_bytes(int d_in, int b_in, int d_out, int b_out) {
  // bf16 K, K^T and G, and fp32 dK, for every block of both sides
  return (2 + 2 + 2 + 4) * ((size_t)d_in * b_in + (size_t)d_out * b_out);
}

namespace {

template <int B>
poetx_status cnp_bwd_ring_launch(const Side& s0, const Side& s1, int n, cudaStream_t s) {
  const int nb = s0.nb + s1.nb;
  CUtensorMap tk0, tg0, tt0, tk1, tg1, tt1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const Side& t0 = s0.nb > 0 ? s0 : s1;
  const Side& t1 = s1.nb > 0 ? s1 : s0;
  if (!make_tmap_2d(&tk0, t0.Kd, bf, 2, (uint64_t)t0.nb * B, B, B, 64, sw) ||
      !make_tmap_2d(&tg0, t0.Gd, bf, 2, (uint64_t)t0.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tt0, t0.Td, bf, 2, (uint64_t)t0.nb * B, B, 128, 64, sw) ||
      !make_tmap_2d(&tk1, t1.Kd, bf, 2, (uint64_t)t1.nb * B, B, B, 64, sw) ||
      !make_tmap_2d(&tg1, t1.Gd, bf, 2, (uint64_t)t1.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tt1, t1.Td, bf, 2, (uint64_t)t1.nb * B, B, 128, 64, sw))
    return POETX_ERR_CUDA;
  constexpr int a_bytes = 128 * B * 2, i_bytes = 128 * 128 * 2, chunk_bytes = B * 64 * 2;
  constexpr int fixed = 2 * a_bytes + i_bytes + 1024 + 256;
  int stages = (kSmemMax - fixed) / chunk_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  const int smem = fixed + stages * chunk_bytes;
  auto kern = cnp_bwd_ring_kernel<B>;
  set_max_dynamic_smem((const void*)kern, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B / 128, nb);
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = B / 128;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int* err = device_error_word();
  {
    KernelScope ks_("tc_cnp_bwd", s);
    if (cudaLaunchKernelEx(&cfg, kern, tk0, tg0, tt0, tk1, tg1, tt1, s0, s1, n, stages, err) !=
        cudaSuccess)
      return check_launch();
  }
  return check_launch();
}

// narrow: the two-CTA ring form (beside a kernel that holds most SMs), else
// the cluster form (b/128 * b/64 CTAs per block).
template <int B>
poetx_status cnp_bwd_launch(const Side& s0, const Side& s1, int n, cudaStream_t s, int parts = 7,
                            bool narrow = false) {
  const int nb = s0.nb + s1.nb;
  if (parts & (kPrepK | kPrepG)) {
    {
      KernelScope ks_("tc_cnp_bwd_prep", s);
      const int z = (parts & kPrepG) ? kPrepZ : 1;   // K alone: one CTA per row group
      cnp_prep_kernel<B><<<dim3(B / kPrepRows, nb, z), kPrepThreads, 0, s>>>(s0, s1, parts & (kPrepK | kPrepG));
    }
    const poetx_status st = check_launch();
    if (st != POETX_OK || !(parts & kChain)) return st;
  }
  if (narrow) return cnp_bwd_ring_launch<B>(s0, s1, n, s);
  CUtensorMap tk0, tg0, tk1, tg1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const Side& t0 = s0.nb > 0 ? s0 : s1;
  const Side& t1 = s1.nb > 0 ? s1 : s0;
  if (!make_tmap_2d(&tk0, t0.Kd, bf, 2, (uint64_t)t0.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tg0, t0.Gd, bf, 2, (uint64_t)t0.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tk1, t1.Kd, bf, 2, (uint64_t)t1.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tg1, t1.Gd, bf, 2, (uint64_t)t1.nb * B, B, 64, 64, sw))
    return POETX_ERR_CUDA;
  using Geo = BwdGeo<B>;
  auto kern = cnp_bwd_kernel<B>;
  set_max_dynamic_smem((const void*)kern, Geo::smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Geo::CL * nb);
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = Geo::smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = Geo::CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int* err = device_error_word();
  {
    KernelScope ks_("tc_cnp_bwd", s);
    if (cudaLaunchKernelEx(&cfg, kern, tk0, tg0, tk1, tg1, s0, s1, n, err) != cudaSuccess)
      return check_launch();
  }
  return check_launch();
}

template <int B>
poetx_status cnp_bwd_sides(const Side& s0, const Side& s1, int n, cudaStream_t s) {
  return cnp_bwd_launch<B>(s0, s1, n, s);
}

poetx_status cnp_bwd_one(const Side& sd, int b, int n, cudaStream_t s, int parts = 7,
                         bool narrow = false) {
  Side none = sd;
  none.nb = 0;
  return b == 256 ? cnp_bwd_launch<256>(sd, none, n, s, parts, narrow)
                  : cnp_bwd_launch<128>(sd, none, n, s, parts, narrow);
}

// The side's part of the workspace: K, K^T, G (bf16) and dK (fp32) of nb blocks.
Side carve(const float* theta, const float* dQ, int n_part, float* dtheta, int nb, int b,
           uint8_t*& w) {
  const size_t e = (size_t)nb * b * b;
  Side sd;
  sd.theta = theta;
  sd.dQ = dQ;
  sd.n_part = n_part;
  sd.dtheta = dtheta;
  sd.nb = nb;
  sd.Kd = reinterpret_cast<__nv_bfloat16*>(w);
  sd.Td = sd.Kd + e;
  sd.Gd = sd.Td + e;
  sd.dK = reinterpret_cast<float*>(sd.Gd + e);
  w += 10 * e;
  return sd;
}

}  // namespace

poetx_status cnp_bwd_side(const float* theta, const float* dQ, int splits, int nb, int b, int n,
                          float* dtheta, void* ws, cudaStream_t s, int parts, bool narrow) {
  if (!cnp_supported(b) || n < 1 || nb > 65535 || splits < 1 || parts < 1 || parts > 7)
    return POETX_ERR_UNSUPPORTED;
  if (nb <= 0) return POETX_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return cnp_bwd_one(carve(theta, dQ, splits, dtheta, nb, b, w), b, n, s, parts, narrow);
}

int cnp_bwd_ctas(int nb, int b) { return nb * (b / 128); }

poetx_status cnp_bwd_layer(const float* theta_P, const float* dQ_P, int splits_P, int nb_P, int b_P,
                           const float* theta_R, const float* dQ_R, int splits_R, int nb_R, int b_R,
                           int n, float* dtheta_P, float* dtheta_R, void* ws, cudaStream_t s) {
  if (!cnp_supported(b_P) || !cnp_supported(b_R) || n < 1 || nb_P + nb_R > 65535 ||
      splits_P < 1 || splits_R < 1)
    return POETX_ERR_UNSUPPORTED;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const Side sp = carve(theta_P, dQ_P, splits_P, dtheta_P, nb_P, b_P, w);
  const Side sr = carve(theta_R, dQ_R, splits_R, dtheta_R, nb_R, b_R, w);
  if (b_P == b_R)
    return b_P == 256 ? cnp_bwd_sides<256>(sp, sr, n, s) : cnp_bwd_sides<128>(sp, sr, n, s);
  const poetx_status st = cnp_bwd_one(sp, b_P, n, s);
  if (st != POETX_OK) return st;
  return cnp_bwd_one(sr, b_R, n, s);
}

}  // namespace tc
}  // namespace poetx
