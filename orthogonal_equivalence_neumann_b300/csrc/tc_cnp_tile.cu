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
// two, b = 128: one); the off-diagonal zeros stay exactly zero through every
// product, so each block is computed as if alone.  The chain is the Horner
// form of Q - I = 2K + 2K^2 + ... + 2K^n + K^{n+1}:
//   X_1 = K,  X_{i+1} = X_i K + 2K  (i = 1..n),  Q = I + X_{n+1},
// each product one tcgen05.mma chain (M = 128 rows, N = 128, K = 16; fp32
// accumulation in TMEM); the 2K term is added in fp32, from the operand's
// own bf16 K (bf16 Q) or its hi + lo parts (fp32 Q), when the accumulator is
// turned into the next operand.
//   bf16 Q:  operands rounded to bf16 (X_i and K);
//   fp32 Q:  every operand split into two bf16 parts, x = hi + lo with
//            hi = bf16(x), lo = bf16(x - hi), and each product taken as
//            X_hi K_hi + X_hi K_lo + X_lo K_hi (the lo * lo term, 2^-16 of
//            the product, is dropped) -- three MMA chains per step; this
//            keeps about 16 significant bits per operand (relative error
//            of Q below 1e-6 at the sweep's sizes, against the fp32 bar of
//            1e-5).
// Operands: B[k][c] = K[k][c], stored as S = -K = K^T (row c of S is column
// c of K), K-major with the 128-byte swizzle, in shared memory; the first
// product reads A = X_1 = K as the same S through a transposed (MN-major)
// descriptor; later products read A = X_i from tensor memory (lane = row,
// two bf16 of consecutive columns per 32-bit column), where the conversion
// of the accumulator writes it.  Thread (warp w, lane l) owns row
// r = 32 (w % 4) + l (its TMEM lane) and half w / 4 of the row's block
// columns.  Tiles are handed out round-robin; one parameter buffer, whose
// next tile's copy is issued as soon as the unpack has read it, so the copy
// runs beside the chain.  Two CTAs share an SM (tensor memory: 256 columns
// each), so one's unpack and conversions overlap the other's products.  One
// thread polls each barrier and the CTA follows through a CTA barrier; every
// wait is bounded (tc_ptx.cuh).
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"

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

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// hi = bf16(v), lo = bf16(v - hi) as 16-bit patterns.
__device__ __forceinline__ void split_bf16(float v, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  hi = (uint32_t)__bfloat16_as_ushort(h);
  lo = bf16_bits(v - __bfloat162float(h));
}

// 8 bf16 of a 16-byte shared-memory unit, widened.
__device__ __forceinline__ void widen8(const uint8_t* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[2 * e] = __uint_as_float(w[e] << 16);
    v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

template <int B, bool F32>
struct TileGeo {
  static constexpr int G = 128 / B;
  static constexpr int P = B * (B - 1) / 2;
  static constexpr int NB32 = B / 32;                      // 32-wide strips of a block
  static constexpr int NOFF = NB32 * (NB32 - 1) / 2;       // pieces above a block's diagonal
  static constexpr int NSUB = G * (NOFF + NB32);           // 32 x 32 pieces unpacked per tile
  static constexpr int n_s = F32 ? 2 : 1;                  // S hi [lo]
  static constexpr int th_bytes = ((G * P * 4 + 127) / 128) * 128;
  static constexpr int used = 1024 + n_s * kOpBytes + th_bytes + 64;
  // two CTAs per SM, as many as tensor memory holds: with less shared memory
  // than 3 x (77 KB + 1 KB) a third CTA could be placed and wait on its
  // allocation
  static constexpr int smem = used > 78848 ? used : 78848;
  static constexpr int per_sm = 2;
  static constexpr int tmem_cols = 256;                    // accumulator 128, X hi 64 [, X lo 64]
};

// Unpack piece `sb` of a tile into S = -K (K-major, 128-byte swizzle) from the
// tile's parameters in shared memory.  Pieces are 32 x 32 parts of a block on
// or above its diagonal, those strictly above first.  Lane l owns column
// j = 32 J + l of the piece (I, J): it reads theta(i, j), i = 32 I .. 32 I + 31
// (a row's parameters are consecutive, so the 32 lanes read one contiguous
// run: no bank conflicts), writes row j of S across the piece's columns
// (S[j][i] = K[i][j] = theta(i, j): four 16-byte stores) and then the column's
// own entries S[i][j] = -theta(i, j) one by one.  In a piece on the diagonal
// the row stores put zeros right of the diagonal and the column stores,
// ordered after them, fill those.  A block the tile does not hold (last
// tile) is written as zeros.
template <int B, bool F32>
__device__ __forceinline__ void unpack_sub(int sb, const float* th_tile, int nbt, uint8_t* s_hi,
                                          uint8_t* s_lo, int lane) {
  using Geo = TileGeo<B, F32>;
  constexpr int NB32 = Geo::NB32, NOFF = Geo::NOFF, G = Geo::G;
  int gb, I, J;
  if (NOFF > 0 && sb < G * NOFF) {
    constexpr int NO = NOFF > 0 ? NOFF : 1;
    gb = sb / NO;
    int q = sb % NO;
    I = 0;
    while (q >= NB32 - 1 - I) {
      q -= NB32 - 1 - I;
      ++I;
    }
    J = I + 1 + q;
  } else {
    const int d = sb - G * NOFF;
    gb = d / NB32;
    I = J = d % NB32;
  }
  const bool live = gb < nbt;
  const int aI = 32 * I, jj = 32 * J + lane;   // first row of the piece, this lane's column
  const float* th = th_tile + (live ? gb : 0) * Geo::P;
  // theta(i, j) sits at skew_row_off(i) + j - i - 1; step the row offset
  // along i: skew_row_off(i + 1) - skew_row_off(i) = B - i - 1
  int idx = skew_row_off(aI, B) + jj - aI - 1;
  uint32_t h[16], l[16];   // theta(aI + r, j) as bf16 pairs (r even in the low half) [hi, lo]
#pragma unroll
  for (int r = 0; r < 32; r += 2) {
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool in = aI + r + e < jj;
      const float t = th[in ? idx : 0];
      v[e] = (live && in) ? t : 0.f;
      idx += B - aI - (r + e) - 2;
    }
    if constexpr (F32) {
      uint32_t h0, l0, h1, l1;
      split_bf16(v[0], h0, l0);
      split_bf16(v[1], h1, l1);
      h[r / 2] = h0 | (h1 << 16);
      l[r / 2] = l0 | (l1 << 16);
    } else {
      h[r / 2] = pack_bf16x2(v[0], v[1]);
    }
  }
  const int R = gb * B + jj;        // this lane's row of the tile (the row stores)
  const int C0 = gb * B + aI;       // first tile column of the piece
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t off = op_off(R, C0 + 8 * q);
    *reinterpret_cast<uint4*>(s_hi + off) =
        make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    if constexpr (F32)
      *reinterpret_cast<uint4*>(s_lo + off) =
          make_uint4(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
  }
  __syncwarp();
  // column stores: S[C0 + r][R] = -theta, the sign bit of each bf16 part
  // flipped (both roundings are symmetric); rows C0 + r share their swizzle
  // phase with r (C0 is a multiple of 32)
  const uint32_t cbase = (uint32_t)((R >> 6) * (128 * 128) + (C0 >> 3) * 1024 + (R & 7) * 2);
  const int cx = (R & 63) >> 3;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    if (aI + r < jj) {
      const uint32_t off = cbase + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((cx ^ (r & 7)) << 4));
      *reinterpret_cast<uint16_t*>(s_hi + off) = (uint16_t)((h[r / 2] >> (16 * (r & 1))) ^ 0x8000u);
      if constexpr (F32)
        *reinterpret_cast<uint16_t*>(s_lo + off) = (uint16_t)((l[r / 2] >> (16 * (r & 1))) ^ 0x8000u);
    }
  }
}

template <int B, bool F32>
__global__ void __launch_bounds__(kTileThreads, 2)
    cnp_tile_kernel(TileSide s0, TileSide s1, int n, int* err) {
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
  const uint32_t x_hi = tmem + 128, x_lo = tmem + 192;  // X_i (i >= 2): [hi, lo] bf16 pairs
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  {
    // X starts at zero too (entries outside the blocks stay so): each thread
    // clears its half of its row
    uint32_t z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = 0;
    tmem_st32(x_hi + lane_off + (uint32_t)(half * 32), z);
    if constexpr (F32) tmem_st32(x_lo + lane_off + (uint32_t)(half * 32), z);
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
      lok = mbar_poll(th_full, (uint32_t)landed & 1, err);
      if (lok) ++landed;
    }
    if (__syncthreads_or(!lok)) {   // every thread leaves together
      ok = false;
      break;
    }

    // ---- unpack S = -K
#pragma unroll 1
    for (int sb = warp; sb < Geo::NSUB; sb += kTileThreads / 32)
      unpack_sub<B, F32>(sb, th_buf, nbt, s_hi, s_lo, lane);
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
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) {   // K = 16 steps
          const uint32_t o = (kq >> 2) * (128 * 128) + (kq & 3) * 32;
          if (i == 1) {
            // A = K = S^T: S read MN-major (its rows are the K index)
            const uint32_t idesc = idesc_bf16(128, 128, true, false);
            const uint32_t oa = kq * (16 * 128);
            mma_bf16(tmem, sw128_desc(sh + oa, 128 * 128, 1024), sw128_desc(sh + o, 16, 1024),
                     idesc, kq != 0);
            if constexpr (F32) {
              mma_bf16(tmem, sw128_desc(sh + oa, 128 * 128, 1024), sw128_desc(sl + o, 16, 1024),
                       idesc, 1);
              mma_bf16(tmem, sw128_desc(sl + oa, 128 * 128, 1024), sw128_desc(sh + o, 16, 1024),
                       idesc, 1);
            }
          } else {
            const uint32_t idesc = idesc_bf16(128, 128, false, false);
            mma_bf16_ts(tmem, x_hi + (uint32_t)(kq * 8), sw128_desc(sh + o, 16, 1024), idesc,
                        kq != 0);
            if constexpr (F32) {
              mma_bf16_ts(tmem, x_hi + (uint32_t)(kq * 8), sw128_desc(sl + o, 16, 1024), idesc, 1);
              mma_bf16_ts(tmem, x_lo + (uint32_t)(kq * 8), sw128_desc(sh + o, 16, 1024), idesc, 1);
            }
          }
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
      // the warp's rows all lie in one block (b >= 32), so its TMEM loads
      // share their columns: [g*B + half*HC, g*B + (half+1)*HC)
#pragma unroll 1
      for (int c0 = half * HC; c0 < (half + 1) * HC; c0 += W) {
        uint32_t acc[W];
        const uint32_t ta = tmem + (uint32_t)(g * B + c0) + lane_off;
        if constexpr (W == 32) tmem_ld32(ta, acc);
        else tmem_ld16(ta, acc);
        // 2K from the operand's own K (S = -K): bf16, or hi + lo for fp32 Q
        float k2[W];
#pragma unroll
        for (int q = 0; q < W / 8; ++q) {
          const uint32_t off = op_off(r, g * B + c0 + 8 * q);
          widen8(s_hi + off, k2 + 8 * q);
          if constexpr (F32) {
            float lo[8];
            widen8(s_lo + off, lo);
#pragma unroll
            for (int e = 0; e < 8; ++e) k2[8 * q + e] += lo[e];
          }
        }
        tmem_ld_wait();
        tmem_regs_ready(acc);
        float x[W];
#pragma unroll
        for (int e = 0; e < W; ++e) x[e] = __uint_as_float(acc[e]) - 2.f * k2[e];
        if (i < n) {
          // X_{i+1} into tensor memory: row r, columns g*B + c0 .. (two per 32-bit column)
          uint32_t h[W / 2], l[W / 2];
#pragma unroll
          for (int e = 0; e < W / 2; ++e) {
            if constexpr (F32) {
              uint32_t h0, l0, h1, l1;
              split_bf16(x[2 * e], h0, l0);
              split_bf16(x[2 * e + 1], h1, l1);
              h[e] = h0 | (h1 << 16);
              l[e] = l0 | (l1 << 16);
            } else {
              h[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
            }
          }
          const uint32_t tx = lane_off + (uint32_t)((g * B + c0) / 2);
          if constexpr (W == 32) {
            tmem_st16(x_hi + tx, h);
            if constexpr (F32) tmem_st16(x_lo + tx, l);
          } else {
            tmem_st8(x_hi + tx, h);
            if constexpr (F32) tmem_st8(x_lo + tx, l);
          }
        } else if (live) {
          // Q = I + X_{n+1}: row ri of block b0 + g
#pragma unroll
          for (int e = 0; e < W; ++e)
            if (c0 + e == ri) x[e] += 1.f;
          const size_t row = ((size_t)(b0 + g) * B + ri) * B + c0;
          if constexpr (F32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(sd->Q) + row);
#pragma unroll
            for (int q = 0; q < W / 4; ++q)
              o[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
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
      tc_fence_before();
      __syncthreads();   // next operand written / S no longer read (the next unpack rewrites it)
    }
    if (!ok) break;
  }
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
  {
    KernelScope ks_(F32 ? "tc_cnp_tile_f32" : "tc_cnp_tile", s);
    cnp_tile_kernel<B, F32><<<grid, kTileThreads, Geo::smem, s>>>(s0, s1, n, device_error_word());
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
