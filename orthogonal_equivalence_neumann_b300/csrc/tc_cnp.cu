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


// ====================================================================== forward
constexpr int kFwdThreads = 288;   // warp 0: TMEM + MMA; warps 1..8: workers
constexpr int kFwdWorkers = 256;

// First packed index of row i (entries (i, i+1) .. (i, b-1)).
__device__ __forceinline__ int skew_row_start(int i, int b) { return (i * (2 * b - i - 1)) >> 1; }

// Row and column of packed index p (the inverse of skew_index): the root of
// the quadratic row-start formula, then an exact integer correction.
__device__ __forceinline__ void skew_rowcol(int p, int b, int& i, int& k) {
  const float t = (float)(2 * b - 1);
  int r = (int)((t - sqrtf(fmaxf(t * t - 8.f * (float)p, 0.f))) * 0.5f);
  r = max(0, min(r, b - 2));
  while (r < b - 2 && skew_row_start(r + 1, b) <= p) ++r;
  while (r > 0 && skew_row_start(r, b) > p) --r;
  i = r;
  k = p - skew_row_start(r, b) + r + 1;
}

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, float v) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(v);
}

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

// One CTA = one 128-row slab of one block.  Shared memory holds Kop, the MMA
// B operand of X -> X K (Kop[c][k] = K[k][c] = -K[c][k], K-major), unpacked
// once from the packed parameters with coalesced 16-byte loads, and the bf16
// A operand X_i of the slab.  The packed parameters are staged again into the
// freed shared memory for the epilogue, which adds the last 2K exactly in fp32.
// Two parameter sets (the P and R factors of a layer) may share a launch:
// blockIdx.y < nb0 selects the first, the rest the second.
struct FwdSide {
  const float* theta;
  void* Q;
  int nb;
};

template <int B>
__global__ void __launch_bounds__(kFwdThreads, 1)
    cnp_fwd_kernel(FwdSide f0, FwdSide f1, int out_f32, int n, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int P = B * (B - 1) / 2;   // packed parameters per block (a multiple of 4)
  uint8_t* kop = smem;                 // [B rows c][B k] bf16
  uint8_t* amat = smem + B * B * 2;    // [128 rows][B k] bf16
  float* ths = reinterpret_cast<float*>(smem);   // epilogue: packed parameters (reuses both)
  uint64_t* afull = reinterpret_cast<uint64_t*>(amat + 128 * B * 2);
  uint64_t* stepdone = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stepdone + 1);
  static_assert(P * 4 <= B * B * 2 + 128 * B * 2, "parameter stage must fit the operands");

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const bool second = (int)blockIdx.y >= f0.nb;
  const int j = second ? (int)blockIdx.y - f0.nb : (int)blockIdx.y;
  void* __restrict__ out = second ? f1.Q : f0.Q;
  const int r0 = blockIdx.x * 128;
  const float* th = (second ? f1.theta : f0.theta) + (size_t)j * P;

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
      const uint32_t ab = smem_u32(amat), bb = smem_u32(kop);
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
    // ---- unpack: Kop[i][k] = -theta(i,k), Kop[k][i] = +theta(i,k), zero diagonal
    {
      const float4* th4 = reinterpret_cast<const float4*>(th);
      constexpr int P4 = P / 4;
      constexpr int BATCH = 8;
      for (int q0 = 0; q0 < P4; q0 += kFwdWorkers * BATCH) {
        float4 v[BATCH];
#pragma unroll
        for (int s = 0; s < BATCH; ++s) {
          const int q = q0 + s * kFwdWorkers + wt;
          if (q < P4) v[s] = __ldg(th4 + q);
        }
#pragma unroll
        for (int s = 0; s < BATCH; ++s) {
          const int q = q0 + s * kFwdWorkers + wt;
          if (q < P4) {
            int i, k;
            skew_rowcol(4 * q, B, i, k);
            const float e4[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              st_bf16(kop, sw128_offset(i, k, B), -e4[e]);
              st_bf16(kop, sw128_offset(k, i, B), e4[e]);
              if (++k == B) { ++i; k = i + 1; }
            }
          }
        }
      }
      for (int c = wt; c < B; c += kFwdWorkers) st_bf16(kop, sw128_offset(c, c, B), 0.f);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kFwdWorkers) : "memory");   // Kop complete
    // ---- X_1 = K on the slab rows: A[r][k] = K[r0+r][k] = -Kop[r0+r][k]
    for (int u = wt; u < 128 * (B / 8); u += kFwdWorkers) {
      const int rr = u / (B / 8), k8 = (u % (B / 8)) * 8;
      uint4 w = *reinterpret_cast<const uint4*>(kop + sw128_offset(r0 + rr, k8, B));
      w.x ^= 0x80008000u; w.y ^= 0x80008000u; w.z ^= 0x80008000u; w.w ^= 0x80008000u;
      *reinterpret_cast<uint4*>(amat + sw128_offset(rr, k8, 128)) = w;
    }
    fence_proxy_async_smem();
    mbar_arrive(afull);
    // ---- X_{i+1} = X_i K + 2K (2K from the bf16 operand; X is rounded to bf16 anyway)
    for (int i = 2; i <= n && ok; ++i) {
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
#pragma unroll
        for (int g = 0; g < 4; ++g)
          *reinterpret_cast<uint4*>(amat + sw128_offset(r, c0 + 8 * g, 128)) = pack8(x + 8 * g);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(afull);
    }
    // ---- epilogue: Q = I + X_n K + 2K, the last 2K exactly from the staged parameters
    if (ok && mbar_wait(stepdone, (n - 1) & 1, err)) {
      tc_fence_after();
      {
        const float4* th4 = reinterpret_cast<const float4*>(th);
        float4* s4 = reinterpret_cast<float4*>(ths);
        for (int q = wt; q < P / 4; q += kFwdWorkers) s4[q] = __ldg(th4 + q);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kFwdWorkers) : "memory");
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rr);
        tmem_ld_wait();
        float q[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int c = c0 + e;
          const float kv = row < c ? ths[skew_index(row, c, B)]
                                   : (row > c ? -ths[skew_index(c, row, B)] : 0.f);
          q[e] = __uint_as_float(rr[e]) + 2.f * kv + (row == c ? 1.f : 0.f);
        }
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
  int nb;
};

constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 32;

// Kd[j] = bf16(K_j), Gd[j] = bf16(dQ_j) for both sides; one CTA per 32-row
// group of one block.  The group's rows of K are assembled in shared memory
// (row pitch B + 2 halves, so the column writes fall in distinct banks):
// entries right of the diagonal come from the packed rows of the group, the
// ones left of it from the packed rows above, which hold the group's columns
// contiguously; both are read with coalesced loads.
template <int B>
__global__ void __launch_bounds__(kPrepThreads)
    cnp_prep_kernel(Side s0, Side s1) {
  __shared__ __nv_bfloat16 tile[kPrepRows * (B + 2)];
  constexpr int LD = B + 2;
  constexpr int P = B * (B - 1) / 2;
  const bool second = (int)blockIdx.y >= s0.nb;
  const Side& sd = second ? s1 : s0;
  const int j = second ? (int)blockIdx.y - s0.nb : (int)blockIdx.y;
  const int c0 = blockIdx.x * kPrepRows;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* th = sd.theta + (size_t)j * P;
  // right of the diagonal: K[c][k] = theta(c, k), packed row c
  for (int rr = warp; rr < kPrepRows; rr += kPrepThreads / 32) {
    const int c = c0 + rr;
    const float* prow = th + skew_row_start(c, B) - (c + 1);   // prow[k] = theta(c, k)
    for (int k = c + 1 + lane; k < B; k += 32) tile[rr * LD + k] = __float2bfloat16_rn(__ldg(prow + k));
    if (lane == 0) tile[rr * LD + c] = __float2bfloat16_rn(0.f);
  }
  // left of the diagonal: K[c][k] = -theta(k, c), packed row k holds columns c0.. contiguously
  for (int k = warp; k < c0 + kPrepRows - 1; k += kPrepThreads / 32) {
    const int c = c0 + lane;
    if (k < c) {
      const float v = __ldg(th + skew_row_start(k, B) + (c - k - 1));
      tile[lane * LD + k] = __float2bfloat16_rn(-v);
    }
  }
  // dQ rows of the group -> bf16
  const float4* g4 = reinterpret_cast<const float4*>(sd.dQ + ((size_t)j * B + c0) * B);
  uint4* gd = reinterpret_cast<uint4*>(sd.Gd + ((size_t)j * B + c0) * B);
  for (int u = threadIdx.x; u < kPrepRows * B / 8; u += kPrepThreads) {
    const float4 a = __ldg(g4 + 2 * u), c = __ldg(g4 + 2 * u + 1);
    gd[u] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(c.x, c.y),
                       pack_bf16x2(c.z, c.w));
  }
  __syncthreads();
  uint32_t* kd = reinterpret_cast<uint32_t*>(sd.Kd + ((size_t)j * B + c0) * B);
  for (int u = threadIdx.x; u < kPrepRows * B / 2; u += kPrepThreads) {
    const int r = u / (B / 2), c2 = (u % (B / 2)) * 2;
    kd[u] = *reinterpret_cast<const uint32_t*>(tile + r * LD + c2);
  }
}

constexpr int kBwdThreads = 320;   // warp 0: TMEM + MMA; warp 1: TMA; warps 2..9: workers
constexpr int kBwdWorkers = 256;

// Bytes of the fp32 dK slab staged for the packing epilogue: 128 rows, stride B + 1.
template <int B>
constexpr int dk_stage_bytes() { return 128 * (B + 1) * 4; }

// One CTA = one 128-row slab of one block; for B = 256 the two slabs of a
// block form a cluster of two CTAs, which exchange the off-diagonal quadrant
// of dK through distributed shared memory when packing dtheta.
template <int B>
__global__ void __launch_bounds__(kBwdThreads, 1)
    cnp_bwd_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tg0,
                   const __grid_constant__ CUtensorMap tk1, const __grid_constant__ CUtensorMap tg1,
                   Side s0, Side s1, int n, int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const bool second = (int)blockIdx.y >= s0.nb;
  const Side& sd = second ? s1 : s0;
  const CUtensorMap* tk = second ? &tk1 : &tk0;
  const CUtensorMap* tg = second ? &tg1 : &tg0;
  const int j = second ? (int)blockIdx.y - s0.nb : (int)blockIdx.y;
  const int slab = blockIdx.x;
  const int r0 = slab * 128;
  constexpr int a_bytes = 128 * B * 2;
  constexpr int chunk_bytes = B * 64 * 2;
  constexpr int kchunks = B / 64;
  constexpr uint32_t ncols = 2 * B;
  constexpr int LDS = B + 1;
  uint8_t* ax = smem;
  uint8_t* ay = smem + a_bytes;
  uint8_t* ring = smem + 2 * a_bytes;
  float* stage = reinterpret_cast<float*>(smem);   // epilogue: dK slab, reuses ax/ay/ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + stages * chunk_bytes);
  uint64_t* bfull = bars;
  uint64_t* bempty = bfull + kMaxStages;
  uint64_t* afull = bempty + kMaxStages;
  uint64_t* stepdone = afull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stepdone + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kMaxStages; ++st) {
      mbar_init(bfull + st, 1);
      mbar_init(bempty + st, 1);
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
  bool ok = true;

  if (warp == 1) {
    // ------------------------------------------------ TMA: per step, K chunks then G^T chunks
    if (lane == 0) {
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
      const uint32_t axb = smem_u32(ax), ayb = smem_u32(ay);
      int st = 0;
      uint32_t ph = 0;
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
    // ------------------------------------------------ workers: A operands, then the dK slab
    const int quarter = warp % 4;
    const int half = (warp - 2) / 4;
    const int r = quarter * 32 + lane;
    const int row = r0 + r;
    const __nv_bfloat16* krow = sd.Kd + ((size_t)j * B + row) * B;   // K[row][.]
    const __nv_bfloat16* gbrow = sd.Gd + ((size_t)j * B + row) * B;  // bf16 G[row][.]
    const float* grow = sd.dQ + ((size_t)j * B + row) * B;           // G[row][.]
    for (int i = 1; i <= n && ok; ++i) {
      if (i > 1) {
        if (!(ok = mbar_wait(stepdone, (i - 2) & 1, err))) break;
        tc_fence_after();
      }
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        float kv[32], gv[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint4 uk = __ldg(reinterpret_cast<const uint4*>(krow + c0 + 8 * g));
          const uint4 ug = __ldg(reinterpret_cast<const uint4*>(gbrow + c0 + 8 * g));
          const uint32_t wk[4] = {uk.x, uk.y, uk.z, uk.w}, wg[4] = {ug.x, ug.y, ug.z, ug.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kv[8 * g + 2 * e] = __uint_as_float(wk[e] << 16);
            kv[8 * g + 2 * e + 1] = __uint_as_float(wk[e] & 0xFFFF0000u);
            gv[8 * g + 2 * e] = __uint_as_float(wg[e] << 16);
            gv[8 * g + 2 * e + 1] = __uint_as_float(wg[e] & 0xFFFF0000u);
          }
        }
        float x[32], y[32];
        if (i == 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = -kv[e];   // K^T[row][c] = -K[row][c]
            y[e] = gv[e];
          }
        } else {
          uint32_t rx[32], ry[32];
          tmem_ld32(tmem_base + (uint32_t)c0 + ((uint32_t)(quarter * 32) << 16), rx);
          tmem_ld32(tmem_base + (uint32_t)(B + c0) + ((uint32_t)(quarter * 32) << 16), ry);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(rx[e]) - 2.f * kv[e];
            y[e] = __uint_as_float(ry[e]) + 2.f * gv[e];
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
    // dK = Y_{n+1} = (last Y product) + 2G, the 2G exactly in fp32; staged in shared memory
    if (ok && (ok = mbar_wait(stepdone, (n - 1) & 1, err))) {
      tc_fence_after();
      for (int c0 = half * (B / 2); c0 < (half + 1) * (B / 2); c0 += 32) {
        uint32_t ry[32];
        tmem_ld32(tmem_base + (uint32_t)(B + c0) + ((uint32_t)(quarter * 32) << 16), ry);
        float g[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(grow + c0) + q);
          g[4 * q] = v.x; g[4 * q + 1] = v.y; g[4 * q + 2] = v.z; g[4 * q + 3] = v.w;
        }
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) stage[r * LDS + c0 + e] = __uint_as_float(ry[e]) + 2.f * g[e];
      }
    }
  }
  // ---- pack: dtheta(i,k) = dK[i][k] - dK[k][i], every packed entry written once.
  // This slab writes the packed rows i of its own slab.  Partner entries
  // dK[k][i] with k in the other slab of the block come from the partner CTA.
  __syncthreads();
  if constexpr (B == 256) cluster_sync();   // both slabs staged
  if (warp >= 2 && ok) {
    const int wt = threadIdx.x - 64;
    const int w8 = wt / 32;
    float* dth = sd.dtheta + (size_t)j * (B * (B - 1) / 2);
    uint32_t partner = 0;
    if constexpr (B == 256) partner = mapa_shared(smem_u32(stage), cluster_ctarank() ^ 1u);
    for (int i = r0 + w8; i < r0 + 128; i += 8) {
      float* drow = dth + skew_index(i, i + 1, B) - (i + 1);   // drow[k] = dtheta(i, k)
      const float* si = stage + (i - r0) * LDS;
      for (int k = i + 1 + lane; k < B; k += 32) {
        float other;
        if (k < r0 + 128) {
          other = stage[(k - r0) * LDS + i];
        } else {
          other = ld_dsmem_f32(partner + (uint32_t)(((k - 128) * LDS + i) * 4));
        }
        drow[k] = si[k] - other;
      }
    }
  }
  if constexpr (B == 256) cluster_sync();   // the partner has finished reading this slab
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ncols);
  }
}

}  // namespace

bool cnp_supported(int b) { return b == 128 || b == 256; }

poetx_status cnp_fwd_pair_bf16ops(const float* theta0, int nb0, const float* theta1, int nb1,
                                  int b, int n, void* Q0, void* Q1, bool out_f32, cudaStream_t s) {
  if (nb0 + nb1 <= 0) return POETX_OK;
  if (!cnp_supported(b) || n < 1 || nb0 + nb1 > 65535) return POETX_ERR_UNSUPPORTED;
  const int smem = b * b * 2 + 128 * b * 2 + 1024 + 256;
  dim3 grid(b / 128, nb0 + nb1);
  FwdSide f0{theta0, Q0, nb0}, f1{theta1, Q1, nb1};
  int* err = device_error_word();
  KernelScope ks_("tc_cnp_fwd", s);
  if (b == 256) {
    cudaFuncSetAttribute(cnp_fwd_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cnp_fwd_kernel<256><<<grid, kFwdThreads, smem, s>>>(f0, f1, out_f32 ? 1 : 0, n, err);
  } else {
    cudaFuncSetAttribute(cnp_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cnp_fwd_kernel<128><<<grid, kFwdThreads, smem, s>>>(f0, f1, out_f32 ? 1 : 0, n, err);
  }
  return check_launch();
}

poetx_status cnp_fwd_bf16ops(const float* theta, int nb, int b, int n, void* Q, bool out_f32,
                             cudaStream_t s) {
  return cnp_fwd_pair_bf16ops(theta, nb, theta, 0, b, n, Q, Q, out_f32, s);
}

size_t cnp_bwd_workspace_bytes(int d_in, int b_in, int d_out, int b_out) {
  // dense bf16 K and bf16 G for every block of both sides
  return 2 * 2 * ((size_t)d_in * b_in + (size_t)d_out * b_out);
}

namespace {

template <int B>
poetx_status cnp_bwd_launch(const Side& s0, const Side& s1, int n, cudaStream_t s) {
  const int nb = s0.nb + s1.nb;
  {
    KernelScope ks_("tc_cnp_bwd_prep", s);
    cnp_prep_kernel<B><<<dim3(B / kPrepRows, nb), kPrepThreads, 0, s>>>(s0, s1);
  }
  poetx_status st = check_launch();
  if (st != POETX_OK) return st;
  CUtensorMap tk0, tg0, tk1, tg1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const Side& t1 = s1.nb > 0 ? s1 : s0;
  if (!make_tmap_2d(&tk0, s0.Kd, bf, 2, (uint64_t)s0.nb * B, B, B, 64, sw) ||
      !make_tmap_2d(&tg0, s0.Gd, bf, 2, (uint64_t)s0.nb * B, B, 64, 64, sw) ||
      !make_tmap_2d(&tk1, t1.Kd, bf, 2, (uint64_t)t1.nb * B, B, B, 64, sw) ||
      !make_tmap_2d(&tg1, t1.Gd, bf, 2, (uint64_t)t1.nb * B, B, 64, 64, sw))
    return POETX_ERR_CUDA;
  constexpr int a_bytes = 128 * B * 2, chunk_bytes = B * 64 * 2;
  int stages = (kSmemMax - 2 * a_bytes - 1024 - 256) / chunk_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  int smem = 2 * a_bytes + stages * chunk_bytes + 1024 + 256;
  if (smem < dk_stage_bytes<B>() + 1024 + 256) smem = dk_stage_bytes<B>() + 1024 + 256;
  auto kern = cnp_bwd_kernel<B>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B / 128, nb);
  cfg.blockDim = dim3(kBwdThreads);
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
    if (cudaLaunchKernelEx(&cfg, kern, tk0, tg0, tk1, tg1, s0, s1, n, stages, err) != cudaSuccess)
      return check_launch();
  }
  return check_launch();
}

template <int B>
poetx_status cnp_bwd_sides(const Side& s0, const Side& s1, int n, cudaStream_t s) {
  return cnp_bwd_launch<B>(s0, s1, n, s);
}

poetx_status cnp_bwd_one(const Side& sd, int b, int n, cudaStream_t s) {
  Side none = sd;
  none.nb = 0;
  return b == 256 ? cnp_bwd_launch<256>(sd, none, n, s) : cnp_bwd_launch<128>(sd, none, n, s);
}

}  // namespace

poetx_status cnp_bwd_layer(const float* theta_P, const float* dQ_P, int nb_P, int b_P,
                           const float* theta_R, const float* dQ_R, int nb_R, int b_R, int n,
                           float* dtheta_P, float* dtheta_R, void* ws, cudaStream_t s) {
  if (!cnp_supported(b_P) || !cnp_supported(b_R) || n < 1 || nb_P + nb_R > 65535)
    return POETX_ERR_UNSUPPORTED;
  __nv_bfloat16* w = static_cast<__nv_bfloat16*>(ws);
  Side sp{theta_P, dQ_P, w, w + (size_t)nb_P * b_P * b_P, dtheta_P, nb_P};
  __nv_bfloat16* w2 = w + 2 * (size_t)nb_P * b_P * b_P;
  Side sr{theta_R, dQ_R, w2, w2 + (size_t)nb_R * b_R * b_R, dtheta_R, nb_R};
  if (b_P == b_R)
    return b_P == 256 ? cnp_bwd_sides<256>(sp, sr, n, s) : cnp_bwd_sides<128>(sp, sr, n, s);
  const poetx_status st = cnp_bwd_one(sp, b_P, n, s);
  if (st != POETX_OK) return st;
  return cnp_bwd_one(sr, b_R, n, s);
}

}  // namespace tc
}  // namespace poetx
