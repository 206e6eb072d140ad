// tc_cnp_tile.cu -- Cayley-Neumann blocks of b <= 128 on the tensor cores,
// unpacked in shared memory.
//
// [POET-X §2.D] ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation", gist.science summary, section 2.D): Q = (I + K)(I + K +
// ... + K^n) for the skew K stored as its upper triangle; the page fuses the
// Neumann chain into one kernel that keeps K and its powers on chip.  Here
// the packed parameters come in by a bulk copy and are unpacked straight into
// shared memory as the MMA operand: the dense K never exists in HBM.
//
// A CTA works on tiles of 128 rows.  A tile holds G = 128 / b consecutive
// blocks as one block-diagonal 128 x 128 matrix (b = 32: four blocks, b = 64:
// two, b = 128: one); each product covers block g's own columns (N = b) from
// its own K range, so the MMA work scales with b and the zeros between the
// blocks are never touched.  The chain is the Horner form of
// Q - I = 2K + 2K^2 + ... + 2K^n + K^{n+1}:
//   X_1 = K,  X_{i+1} = X_i K + 2K  (i = 1..n),  Q = I + X_{n+1},
// each product one tcgen05.mma chain (M = 128 rows, K = 16 per instruction;
// fp32 accumulation in TMEM).
//   bf16 Q:  operands rounded to bf16 (X_i and K); for b >= 64 the 2K term
//            is a second product, 2I . K, into the same accumulator (2I sits
//            in TMEM; 2 * bf16 is exact), so the accumulator is X_{i+1} as
//            it stands; at b = 32 it is added in fp32 from K when the
//            accumulator is read;
//   fp32 Q:  every operand split into two fp16 parts, x = hi + lo with
//            hi = fp16(x), lo = fp16(x - hi), and each product taken as
//            X_hi K_hi + X_hi K_lo + X_lo K_hi (the lo * lo term, 2^-22 of
//            the product, is dropped) -- three MMA chains per step; the 2K
//            term is added in fp32 from K's hi + lo parts when the
//            accumulator is read.  This keeps about 22 significant bits per
//            operand (the lo parts of small entries fall into fp16's
//            subnormal range, about 3e-8 absolute: far below the fp32 bar
//            of 1e-5 relative to Q; bf16 parts, 16 bits, would leave rows
//            of Q some 6e-6 off at sigma = 0.05).
// Operands: B[k][c] = K[k][c], stored as S = -K = K^T (row c of S is column
// c of K), K-major with the 128-byte swizzle, in shared memory; the first
// product reads A = X_1 = K as the same S through a transposed (MN-major)
// descriptor; later products read A = X_i from tensor memory (lane = row,
// two bf16 of consecutive columns per 32-bit column), where the conversion
// of the accumulator writes it.  The unpack turns the packed parameters into
// S with warp-wide 8 x 8 fragment stores (stmatrix, plain and transposed).
// Thread (warp w, lane l) owns row r = 32 (w % 4) + l (its TMEM lane) and
// half w / 4 of the row's block columns.  Q leaves through shared memory
// and tensor stores where its rows fill 128-byte boxes (bf16 Q of b >= 64,
// fp32 Q of b = 128), else by each thread's row stores.  Tiles are handed
// out round-robin; one parameter buffer, whose next tile's bulk copy is
// issued as soon as the unpack has read it, so the copy runs beside the
// chain.  Two CTAs share an SM (tensor memory: 256 columns each), so one's
// unpack and conversions overlap the other's products.  One thread polls
// each barrier and the CTA follows through a CTA barrier; every wait is
// bounded (tc_ptx.cuh).
#include <cstring>

#include <cuda_fp16.h>

#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int kTileThreads = 256;   // two threads per row of the tile (TMEM lane), one per column half
constexpr int kOpBytes = 128 * 128 * 2;

struct TileSide {
  const float* theta;
  void* Q;
  int nb;
};

__device__ __forceinline__ int skew_row_off(int i, int b) { return (i * (2 * b - i - 1)) >> 1; }

// Byte offset of element (r, k) of a 128 x 128 bf16 operand, K-major, 128-byte swizzle.
__device__ __forceinline__ uint32_t op_off(int r, int k) {
  return (uint32_t)((k >> 6) * (128 * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// hi = fp16(v), lo = fp16(v - hi) as 16-bit patterns (v = hi + lo + e,
// |e| <= 2^-22 |v| above fp16's subnormal range).
__device__ __forceinline__ void split_f16(float v, uint32_t& hi, uint32_t& lo) {
  const __half h = __float2half_rn(v);
  hi = (uint32_t)__half_as_ushort(h);
  lo = (uint32_t)__half_as_ushort(__float2half_rn(v - __half2float(h)));
}

// 8 bf16 of a 16-byte unit, widened.
__device__ __forceinline__ void widen8(const uint4 u, float* v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// 8 fp16 of a 16-byte unit, widened.
__device__ __forceinline__ void widen8_f16(const uint4 u, float* v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

template <int B, bool F32>
struct TileGeo {
  static constexpr int G = 128 / B;
  static constexpr int P = B * (B - 1) / 2;
  static constexpr int NU = B * (B + 32) / 512;            // 8 x 32 unpack units of a block
  static constexpr int NUNITS = G * NU;                    // ... of a tile (b = 128: 40)
  static constexpr int n_s = F32 ? 2 : 1;                  // S hi [lo]
  static constexpr int th_bytes = ((G * P * 4 + 127) / 128) * 128;
  static constexpr int used = 1024 + n_s * kOpBytes + th_bytes + 64;
  // two CTAs per SM, as many as tensor memory holds: with less shared memory
  // than 3 x (77 KB + 1 KB) a third CTA could be placed and wait on its
  // allocation
  static constexpr int smem = used > 78848 ? used : 78848;
  static constexpr int per_sm = 2;
  static constexpr int tmem_cols = 256;                    // accumulator 128, X hi 64 [, X lo 64]
  // Q leaves through shared memory (S, free after the last product) and
  // tensor stores, in 128-byte rows: bf16 Q of b >= 64 (as the operand
  // layout), fp32 Q of b = 128 (32-column boxes over S's rows)
  static constexpr bool staged_out = (!F32 && B >= 64) || (F32 && B == 128);
  // bf16 Q of b >= 64 takes the 2K term as a product with 2I (at b = 32 the
  // conversion's share of a step is small and the extra MMAs cost more)
  static constexpr bool two_i_mma = !F32 && B >= 64;
};

// -x for each 16-bit float of a pair that is not zero (bf16 or fp16: the sign
// is bit 15; zeros keep their +0 pattern).
__device__ __forceinline__ uint32_t neg_nonzero(uint32_t h) {
  return h ^ (((h & 0x7fff7fffu) + 0x7fff7fffu) & 0x80008000u);
}

// Unpack unit `u` of a tile into S = -K (K-major, 128-byte swizzle) from the
// tile's parameters in shared memory.  A unit is 8 rows x 32 columns of a
// block, rows [8 I, 8 I + 8), columns [32 J, 32 J + 32), holding at least one
// entry above the diagonal (8 I < 32 J + 32): 2 J (J + 1) units of strip J
// come before strip J + 1, so a block of b has b (b + 32) / 512 of them
// (b = 128: 40, five per warp).  The warp holds the unit as four 8 x 8
// fragments M_q = theta(8 I + r, 32 J + 8 q + c) (zero on and below the
// diagonal) and writes each twice with stmatrix: S over rows 8 I.., columns
// 32 J + 8 q.. is -M_q, S over rows 32 J + 8 q.., columns 8 I.. is M_q^T.
// The fragment on the diagonal (8 q = 8 I - 32 J) holds both halves of one
// 8 x 8 part of S, -M + M^T, built in registers and written once; fragments
// left of it lie below the diagonal (other units' transposed writes cover
// those parts).  So every 8 x 8 part of a block is written exactly once per
// tile; a block the tile does not hold (last tile) is written as zeros.
template <int B, bool F32>
__device__ __forceinline__ void unpack_unit(int u, const float* th_tile, int nbt, uint32_t s_hi,
                                           uint32_t s_lo, int lane) {
  using Geo = TileGeo<B, F32>;
  const int gb = u / Geo::NU;
  const int w = u % Geo::NU;
  int J = 0;
  while (2 * (J + 1) * (J + 2) <= w) ++J;
  const int I = w - 2 * J * (J + 1);
  const bool live = gb < nbt;
  const int a = 8 * I;                    // first row of the unit (block-relative)
  const int qd = (a - 32 * J) >> 3;       // the fragment on the diagonal (< 0: none)
  // this lane's fragment entries: row a + lane / 4, columns 32 J + 8 q + cp + {0, 1};
  // theta(i, j) sits at skew_row_off(i) + j - i - 1
  const int i = a + (lane >> 2), cp = 2 * (lane & 3);
  const float* th = th_tile + (live ? gb : 0) * Geo::P + (skew_row_off(i, B) - i - 1 + 32 * J + cp);
  uint32_t h[4], l[4];   // M_q as 16-bit pairs: bf16, or fp16 [hi, lo] parts for fp32 Q
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool in = live && q >= qd && (q > qd || i < 32 * J + 8 * q + cp + e);
      v[e] = in ? th[8 * q + e] : 0.f;
    }
    if constexpr (F32) {
      uint32_t h0, l0, h1, l1;
      split_f16(v[0], h0, l0);
      split_f16(v[1], h1, l1);
      h[q] = h0 | (h1 << 16);
      l[q] = l0 | (l1 << 16);
    } else {
      h[q] = pack_bf16x2(v[0], v[1]);
    }
  }
  const int t8 = lane & 7, m = lane >> 3;   // the row this lane addresses, of fragment m
  const int base = gb * B;
  if (qd < 0) {
    // every fragment above the diagonal
    const uint32_t dir = op_off(base + a + t8, base + 32 * J + 8 * m);
    const uint32_t tr = op_off(base + 32 * J + 8 * m + t8, base + a);
    stmatrix_x4(s_hi + dir, neg_nonzero(h[0]), neg_nonzero(h[1]), neg_nonzero(h[2]),
                neg_nonzero(h[3]));
    stmatrix_x4_trans(s_hi + tr, h[0], h[1], h[2], h[3]);
    if constexpr (F32) {
      stmatrix_x4(s_lo + dir, neg_nonzero(l[0]), neg_nonzero(l[1]), neg_nonzero(l[2]),
                  neg_nonzero(l[3]));
      stmatrix_x4_trans(s_lo + tr, l[0], l[1], l[2], l[3]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q < qd) continue;
      const uint32_t dir = op_off(base + a + t8, base + 32 * J + 8 * q);
      if (q == qd) {
        // -M + M^T: where one is non-zero the other is zero
        stmatrix_x1(s_hi + dir, movmatrix_trans(h[q]) | neg_nonzero(h[q]));
        if constexpr (F32) stmatrix_x1(s_lo + dir, movmatrix_trans(l[q]) | neg_nonzero(l[q]));
      } else {
        const uint32_t tr = op_off(base + 32 * J + 8 * q + t8, base + a);
        stmatrix_x1(s_hi + dir, neg_nonzero(h[q]));
        stmatrix_x1_trans(s_hi + tr, h[q]);
        if constexpr (F32) {
          stmatrix_x1(s_lo + dir, neg_nonzero(l[q]));
          stmatrix_x1_trans(s_lo + tr, l[q]);
        }
      }
    }
  }
}

template <int B, bool F32>
__global__ void __launch_bounds__(kTileThreads, 2)
    cnp_tile_kernel(TileSide s0, TileSide s1, const __grid_constant__ CUtensorMap tq0,
                    const __grid_constant__ CUtensorMap tq1, int staged, int n, int* err) {
  using Geo = TileGeo<B, F32>;
  constexpr int G = Geo::G, P = Geo::P;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* s_hi = smem;                                    // S = -K (bf16 hi part)
  uint8_t* s_lo = smem + kOpBytes;                         // (fp32 only) lo part
  float* th_buf = reinterpret_cast<float*>(smem + Geo::n_s * kOpBytes);
  uint64_t* th_full = reinterpret_cast<uint64_t*>(smem + Geo::n_s * kOpBytes + Geo::th_bytes);
  uint64_t* mma_done = th_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4, half = warp / 4;
  const int r = quarter * 32 + lane;        // row of the tile = TMEM lane
  const int g = r / B, ri = r % B;          // block of the tile, row within it
  const int tiles0 = (s0.nb + G - 1) / G, tiles1 = (s1.nb + G - 1) / G;
  const int tiles = tiles0 + tiles1;
  const bool leader = threadIdx.x == 0;

  // S starts at zero: entries outside the tile's blocks are never written
  for (int o = threadIdx.x * 16; o < Geo::n_s * kOpBytes; o += kTileThreads * 16)
    *reinterpret_cast<uint4*>(smem + o) = make_uint4(0, 0, 0, 0);
  if (leader) {
    mbar_init(th_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, Geo::tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;                     // accumulator: columns [0, 128)
  const uint32_t x_hi = tmem + 128;                     // X_i (i >= 2): bf16 pairs [hi part]
  const uint32_t x_lo = tmem + 192;                     // fp32 Q: X_i lo part
  const uint32_t two_i = tmem + 192;                    // bf16 Q: 2I, the A of the 2K term
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  {
    // X starts at zero too (entries outside the blocks stay so); each thread
    // writes its half of its row
    uint32_t z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = 0;
    tmem_st32(x_hi + lane_off + (uint32_t)(half * 32), z);
    if constexpr (F32) {
      tmem_st32(x_lo + lane_off + (uint32_t)(half * 32), z);
    } else if constexpr (Geo::two_i_mma) {
      // 2I: 2.0 (bf16 0x4000) at column r of row r
      uint32_t d2[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        d2[e] = half * 32 + e == r / 2 ? ((r & 1) ? 0x40000000u : 0x00004000u) : 0u;
      tmem_st32(two_i + lane_off + (uint32_t)(half * 32), d2);
    }
    tmem_st_wait();
  }

  // tile t -> side, first block, blocks in the tile
  auto locate = [&](int t, const TileSide*& sd, int& b0, int& nbt) {
    const bool second = t >= tiles0;
    sd = second ? &s1 : &s0;
    b0 = (second ? t - tiles0 : t) * G;
    nbt = min(G, sd->nb - b0);
  };
  auto fetch = [&](int t) {   // the tile's parameters, one bulk copy
    const TileSide* sd;
    int b0, nbt;
    locate(t, sd, b0, nbt);
    const uint32_t bytes = (uint32_t)(nbt * P * 4);   // a multiple of 16 for b >= 32
    mbar_arrive_expect_tx(th_full, bytes);
    bulk_load_g2s(th_buf, sd->theta + (size_t)b0 * P, bytes, th_full);
  };

  bool ok = true, mma_pending = false;
  uint32_t mma_count = 0;
  int fetched = 0, landed = 0;   // parameter copies issued / waited for (leader)
  if (leader && (int)blockIdx.x < tiles) {
    fetch(blockIdx.x);
    fetched = 1;
  }
  // this thread's columns of its row: half `half` of the block's B columns
  constexpr int HC = B / 2;
  constexpr int W = HC < 32 ? HC : 32;   // columns per TMEM load
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const TileSide* sd;
    int b0, nbt;
    locate(t, sd, b0, nbt);
    const bool live = g < nbt;   // rows of a missing block (last tile) stay zero
    bool lok = true;
    if (leader) {
      // the last tile's output stores have read S before the unpack rewrites it
      if (Geo::staged_out && staged) bulk_wait_read0();
      lok = mbar_poll(th_full, (uint32_t)landed & 1, err);
      if (lok) ++landed;
    }
    if (__syncthreads_or(!lok)) {   // every thread leaves together
      ok = false;
      break;
    }

    // ---- unpack S = -K
#pragma unroll 1
    for (int u = warp; u < Geo::NUNITS; u += kTileThreads / 32)
      unpack_unit<B, F32>(u, th_buf, nbt, smem_u32(s_hi), smem_u32(s_lo), lane);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // the parameter buffer is read: the next tile's copy runs beside the chain
    if (leader && t + (int)gridDim.x < tiles) {
      fence_proxy_async_smem();
      fetch(t + (int)gridDim.x);
      ++fetched;
    }

    // ---- the chain
    for (int i = 1; i <= n; ++i) {
      lok = true;
      if (leader) {
        tc_fence_after();
        const uint32_t sh = smem_u32(s_hi), sl = smem_u32(s_lo);
        // block-diagonal products: block gq's output columns (N = B) from
        // its own K range only (the rest of X's rows there are zero)
        // fp32 Q: the operands' parts are fp16
        const uint32_t id_kk = F32 ? idesc_f16(128, B, false, false) : idesc_bf16(128, B, false, false);
        const uint32_t id_mk = F32 ? idesc_f16(128, B, true, false) : idesc_bf16(128, B, true, false);
        // descriptors of S at an offset: the start-address field of the base
        // descriptor plus offset / 16 (shared addresses stay below 2^18, so
        // the 14-bit field never carries)
        const uint64_t dk_h = sw128_desc(sh, 16, 1024), dk_l = sw128_desc(sl, 16, 1024);
        const uint64_t dm_h = sw128_desc(sh, 128 * 128, 1024), dm_l = sw128_desc(sl, 128 * 128, 1024);
#pragma unroll
        for (int gq = 0; gq < G; ++gq)
#pragma unroll
          for (int kq = 0; kq < B / 16; ++kq) {   // K = 16 steps
            const int k0 = gq * B + 16 * kq;
            const uint32_t d = tmem + (uint32_t)(gq * B);
            const uint32_t ob =
                (uint32_t)((k0 >> 6) * (128 * 128) + gq * B * 128 + ((k0 & 63) >> 4) * 32);
            const uint32_t acc0 = kq != 0;
            if (i == 1) {
              // A = K = S^T: S read MN-major (its rows are the K index)
              const uint32_t oa = (uint32_t)(k0 * 128);
              mma_bf16(d, dm_h + (oa >> 4), dk_h + (ob >> 4), id_mk, acc0);
              if constexpr (F32) {
                mma_bf16(d, dm_h + (oa >> 4), dk_l + (ob >> 4), id_mk, 1);
                mma_bf16(d, dm_l + (oa >> 4), dk_h + (ob >> 4), id_mk, 1);
              }
            } else {
              const uint32_t xa = (uint32_t)(k0 / 2);
              mma_bf16_ts(d, x_hi + xa, dk_h + (ob >> 4), id_kk, acc0);
              if constexpr (F32) {
                mma_bf16_ts(d, x_hi + xa, dk_l + (ob >> 4), id_kk, 1);
                mma_bf16_ts(d, x_lo + xa, dk_h + (ob >> 4), id_kk, 1);
              }
            }
            if constexpr (Geo::two_i_mma)   // + 2I . K
              mma_bf16_ts(d, two_i + (uint32_t)(k0 / 2), dk_h + (ob >> 4), id_kk, 1);
          }
        mma_commit(mma_done);
        lok = mbar_poll(mma_done, mma_count & 1, err);
      }
      if (__syncthreads_or(!lok)) {
        ok = false;
        mma_pending = true;
        break;
      }
      ++mma_count;
      tc_fence_after();
      // fp32 Q staged (b = 128): the output's first 32 columns go over this
      // thread's row of S lo, the second over its row of S hi (no other
      // thread reads those bytes); the lo part the second pass needs is read
      // before the first overwrites it
      const bool stage_f32 = F32 && Geo::staged_out && staged && i == n;
      uint4 lo_next[4];
      if (stage_f32) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          lo_next[q] = *reinterpret_cast<const uint4*>(s_lo + op_off(r, half * HC + 32 + 8 * q));
      }
      // the warp's rows all lie in one block (b >= 32), so its TMEM loads
      // share their columns: [g*B + half*HC, g*B + (half+1)*HC)
#pragma unroll 1
      for (int c0 = half * HC; c0 < (half + 1) * HC; c0 += W) {
        uint32_t acc[W];
        const uint32_t ta = tmem + (uint32_t)(g * B + c0) + lane_off;
        if constexpr (W == 32) tmem_ld32(ta, acc);
        else tmem_ld16(ta, acc);
        float x[W];
        if constexpr (!Geo::two_i_mma) {
          // 2K from the operand's own K (S = -K): bf16, or hi + lo for fp32 Q
          float k2[W];
#pragma unroll
          for (int q = 0; q < W / 8; ++q) {
            const uint32_t off = op_off(r, g * B + c0 + 8 * q);
            if constexpr (F32) {
              float lo[8];
              widen8_f16(*reinterpret_cast<const uint4*>(s_hi + off), k2 + 8 * q);
              widen8_f16(stage_f32 && c0 != half * HC ? lo_next[q]
                                                      : *reinterpret_cast<const uint4*>(s_lo + off),
                         lo);
#pragma unroll
              for (int e = 0; e < 8; ++e) k2[8 * q + e] += lo[e];
            } else {
              widen8(*reinterpret_cast<const uint4*>(s_hi + off), k2 + 8 * q);
            }
          }
          tmem_ld_wait();
          tmem_regs_ready(acc);
#pragma unroll
          for (int e = 0; e < W; ++e) x[e] = __uint_as_float(acc[e]) - 2.f * k2[e];
        } else {
          // the products already hold the 2K term
          tmem_ld_wait();
          tmem_regs_ready(acc);
#pragma unroll
          for (int e = 0; e < W; ++e) x[e] = __uint_as_float(acc[e]);
        }
        if (i < n) {
          // X_{i+1} into tensor memory: row r, columns g*B + c0 .. (two per 32-bit column)
          uint32_t h[W / 2], l[W / 2];
          float big = 0.f;
#pragma unroll
          for (int e = 0; e < W / 2; ++e) {
            if constexpr (F32) {
              uint32_t h0, l0, h1, l1;
              split_f16(x[2 * e], h0, l0);
              split_f16(x[2 * e + 1], h1, l1);
              h[e] = h0 | (h1 << 16);
              l[e] = l0 | (l1 << 16);
              big = fmaxf(big, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
            } else {
              h[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
            }
          }
          if (F32 && big >= 65504.f) raise_device_error(err, POETX_ERR_RANGE);   // beyond fp16
          const uint32_t tx = lane_off + (uint32_t)((g * B + c0) / 2);
          if constexpr (W == 32) {
            tmem_st16(x_hi + tx, h);
            if constexpr (F32) tmem_st16(x_lo + tx, l);
          } else {
            tmem_st8(x_hi + tx, h);
            if constexpr (F32) tmem_st8(x_lo + tx, l);
          }
        } else if (live) {
          // Q = I + X_{n+1}: row ri of block b0 + g (the diagonal lies in
          // these columns for all or none of most warps' lanes)
          if (__any_sync(0xffffffffu, (unsigned)(ri - c0) < (unsigned)W)) {
#pragma unroll
            for (int e = 0; e < W; ++e)
              if (c0 + e == ri) x[e] += 1.f;
          }
          const size_t row = ((size_t)(b0 + g) * B + ri) * B + c0;
          if constexpr (F32) {
            if (stage_f32) {
              // a 128-row x 32-column fp32 box, 128-byte swizzle: row r's
              // 16-byte chunk q at r * 128 + (q ^ (r % 8)) * 16
              uint8_t* dst = (c0 == half * HC ? s_lo : s_hi) + half * (128 * 128) + r * 128;
#pragma unroll
              for (int q = 0; q < W / 4; ++q)
                *reinterpret_cast<float4*>(dst + ((q ^ (r & 7)) << 4)) =
                    make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            } else {
              float4* o = reinterpret_cast<float4*>(static_cast<float*>(sd->Q) + row);
#pragma unroll
              for (int q = 0; q < W / 4; ++q)
                o[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            }
          } else if (Geo::staged_out && staged) {
            // into S (free: the products are done and bf16 Q reads no K here)
#pragma unroll
            for (int q = 0; q < W / 8; ++q)
              *reinterpret_cast<uint4*>(s_hi + op_off(r, g * B + c0 + 8 * q)) =
                  make_uint4(pack_bf16x2(x[8 * q], x[8 * q + 1]),
                             pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                             pack_bf16x2(x[8 * q + 4], x[8 * q + 5]),
                             pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(sd->Q) + row);
#pragma unroll
            for (int q = 0; q < W / 8; ++q)
              o[q] = make_uint4(pack_bf16x2(x[8 * q], x[8 * q + 1]),
                                pack_bf16x2(x[8 * q + 2], x[8 * q + 3]),
                                pack_bf16x2(x[8 * q + 4], x[8 * q + 5]),
                                pack_bf16x2(x[8 * q + 6], x[8 * q + 7]));
          }
        }
      }
      if (i < n) tmem_st_wait();
      else if (Geo::staged_out && staged) fence_proxy_async_smem();   // for the tensor stores
      tc_fence_before();
      __syncthreads();   // next operand written / S no longer read (the next unpack rewrites it)
      if (Geo::staged_out && staged && i == n && leader) {
        // the tile's blocks: 128-byte column halves of S's rows (b = 128),
        // or block g's rows in S's column half g (b = 64)
        const CUtensorMap* tq = sd == &s0 ? &tq0 : &tq1;
        if constexpr (F32) {   // boxes of 32 columns: S lo / S hi rows of column half 0, then 1
          tma_store_2d(tq, s_lo, 0, b0 * B);
          tma_store_2d(tq, s_hi, 32, b0 * B);
          tma_store_2d(tq, s_lo + 128 * 128, 64, b0 * B);
          tma_store_2d(tq, s_hi + 128 * 128, 96, b0 * B);
        } else if constexpr (B == 128) {
          tma_store_2d(tq, s_hi, 0, b0 * B);
          tma_store_2d(tq, s_hi + 128 * 128, 64, b0 * B);
        } else {
          for (int gg = 0; gg < nbt; ++gg)
            tma_store_2d(tq, s_hi + gg * (128 * 128 + 64 * 128), 0, (b0 + gg) * B);
        }
        bulk_commit();
      }
    }
    if (!ok) break;
  }
  if (Geo::staged_out && staged && leader) bulk_wait0();   // output stores complete
  if (!ok && leader) {
    // wind-down after an expired wait: the copies and MMAs already issued
    // finish (bounded waits) before the CTA frees its memory
    for (int k = landed; k < fetched; ++k)
      mbar_wait_bounded(th_full, (uint32_t)k & 1, 1u << 16, nullptr);
    if (mma_pending) mbar_wait_bounded(mma_done, mma_count & 1, 1u << 16, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Geo::tmem_cols);
  }
}

template <int B, bool F32>
poetx_status tile_launch(const TileSide& s0, const TileSide& s1, int n, cudaStream_t s) {
  using Geo = TileGeo<B, F32>;
  const void* kern = (const void*)cnp_tile_kernel<B, F32>;
  if (set_max_dynamic_smem(kern, Geo::smem) != cudaSuccess) return check_launch();
  const int tiles = (s0.nb + Geo::G - 1) / Geo::G + (s1.nb + Geo::G - 1) / Geo::G;
  int grid = device_sm_count() * Geo::per_sm;
  if (grid > tiles) grid = tiles;
  // output tensor maps (rows = blocks x b, b columns; 128-byte boxes); where
  // one cannot be made (an unaligned Q) the kernel stores rows directly
  CUtensorMap tq[2];
  memset(tq, 0, sizeof(tq));
  int staged = Geo::staged_out ? 1 : 0;
  const TileSide* sides[2] = {&s0, &s1};
  for (int k = 0; k < 2 && staged; ++k)
    if (sides[k]->nb > 0 &&
        !(F32 ? make_tmap_2d(&tq[k], sides[k]->Q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                             (uint64_t)sides[k]->nb * B, (uint64_t)B, 128, 32,
                             CU_TENSOR_MAP_SWIZZLE_128B)
              : make_tmap_2d(&tq[k], sides[k]->Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                             (uint64_t)sides[k]->nb * B, (uint64_t)B, B == 128 ? 128 : 64, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B)))
      staged = 0;
  {
    KernelScope ks_(F32 ? "tc_cnp_tile_f32" : "tc_cnp_tile", s);
    cnp_tile_kernel<B, F32><<<grid, kTileThreads, Geo::smem, s>>>(s0, s1, tq[0], tq[1], staged, n,
                                                                  device_error_word());
  }
  return check_launch();
}

template <bool F32>
poetx_status tile_dispatch(int b, const TileSide& s0, const TileSide& s1, int n, cudaStream_t s) {
  switch (b) {
    case 32: return tile_launch<32, F32>(s0, s1, n, s);
    case 64: return tile_launch<64, F32>(s0, s1, n, s);
    case 128: return tile_launch<128, F32>(s0, s1, n, s);
  }
  return POETX_ERR_UNSUPPORTED;
}

}  // namespace

bool cnp_tile_supported(int b) { return b == 32 || b == 64 || b == 128; }

poetx_status cnp_tile_fwd(const float* theta0, int nb0, const float* theta1, int nb1, int b, int n,
                          void* Q0, void* Q1, bool out_f32, cudaStream_t s) {
  if (!cnp_tile_supported(b) || n < 1 || nb0 < 0 || nb1 < 0) return POETX_ERR_UNSUPPORTED;
  if (nb0 + nb1 == 0) return POETX_OK;
  const TileSide t0{theta0, Q0, nb0}, t1{theta1, Q1, nb1};
  return out_f32 ? tile_dispatch<true>(b, t0, t1, n, s) : tile_dispatch<false>(b, t0, t1, n, s);
}

}  // namespace tc
}  // namespace poetx
