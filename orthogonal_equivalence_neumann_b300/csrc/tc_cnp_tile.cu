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
// Operand layout: B[c][k] = K[k][c] = -K[c][k] (the MMA computes A . B^T),
// A[r][k] = X[r][k], both K-major with the 128-byte swizzle.  Thread (warp w,
// lane l) owns row r = 32 (w % 4) + l (its TMEM lane) and half w / 4 of the
// row's block columns.  Tiles are handed out round-robin; the next tile's
// parameters are fetched while the current chain runs (or, where a single
// parameter buffer lets more CTAs share an SM, those CTAs' chains hide each
// other's latency instead).  One thread polls each barrier and the CTA
// follows through a CTA barrier; every wait is bounded (tc_ptx.cuh).
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

template <int B, bool F32>
struct TileGeo {
  static constexpr int G = 128 / B;
  static constexpr int P = B * (B - 1) / 2;
  static constexpr int th_floats = G * P;                 // parameters of one tile
  static constexpr int th_bytes = ((th_floats * 4 + 127) / 128) * 128;
  static constexpr int n_ops = F32 ? 4 : 2;               // B hi [lo], A hi [lo]
  static constexpr int smem_with(int nth) { return 1024 + n_ops * kOpBytes + nth * th_bytes + 64; }
  static constexpr int per_sm(int bytes) { return 232448 / (bytes + 1024); }
  // two parameter buffers (the next tile's parameters arrive during this
  // tile's chain), unless one buffer lets more CTAs share an SM (whose chains
  // then hide each other's latency)
  static constexpr int NTH = per_sm(smem_with(1)) > per_sm(smem_with(2)) ? 1 : 2;
  static constexpr int smem = smem_with(NTH);
};

// K[ri][kl] of one block from its packed parameters in shared memory, without
// branches (so the loads of a group can all be in flight): the entry of the
// upper triangle at (min, max), negated below the diagonal, zero on it.
template <int B>
__device__ __forceinline__ float k_entry(const float* th, int ri, int kl) {
  const int lo = min(ri, kl), hi = max(ri, kl);
  const float v = th[max(skew_row_off(lo, B) + (hi - lo - 1), 0)];
  return ri == kl ? 0.f : (ri < kl ? v : -v);
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
__global__ void __launch_bounds__(kTileThreads)
    cnp_tile_kernel(TileSide s0, TileSide s1, int n, int* err) {
  using Geo = TileGeo<B, F32>;
  constexpr int G = Geo::G, P = Geo::P;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* b_hi = smem;                                    // B = -K (bf16 hi part)
  uint8_t* b_lo = smem + kOpBytes;                         // (fp32 only) lo part
  uint8_t* a_hi = smem + (F32 ? 2 : 1) * kOpBytes;         // A = X_i
  uint8_t* a_lo = smem + 3 * kOpBytes;                     // (fp32 only)
  float* th_buf = reinterpret_cast<float*>(smem + Geo::n_ops * kOpBytes);   // [NTH][th_bytes]
  uint64_t* th_full = reinterpret_cast<uint64_t*>(smem + Geo::n_ops * kOpBytes + Geo::NTH * Geo::th_bytes);
  uint64_t* mma_done = th_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4, half = warp / 4;
  const int r = quarter * 32 + lane;        // row of the tile = TMEM lane
  const int g = r / B, ri = r % B;          // block of the tile, row within it
  const int tiles0 = (s0.nb + G - 1) / G, tiles1 = (s1.nb + G - 1) / G;
  const int tiles = tiles0 + tiles1;
  const bool leader = threadIdx.x == 0;

  if (leader) {
    mbar_init(th_full, 1);
    mbar_init(th_full + 1, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // tile t -> side, first block, blocks in the tile
  auto locate = [&](int t, const TileSide*& sd, int& b0, int& nbt) {
    const bool second = t >= tiles0;
    sd = second ? &s1 : &s0;
    b0 = (second ? t - tiles0 : t) * G;
    nbt = min(G, sd->nb - b0);
  };
  auto fetch = [&](int t, int buf) {   // the tile's parameters, one bulk copy
    const TileSide* sd;
    int b0, nbt;
    locate(t, sd, b0, nbt);
    const uint32_t bytes = (uint32_t)(nbt * P * 4);   // a multiple of 16 for b >= 32
    mbar_arrive_expect_tx(th_full + buf, bytes);
    bulk_load_g2s(reinterpret_cast<uint8_t*>(th_buf) + buf * Geo::th_bytes,
                  sd->theta + (size_t)b0 * P, bytes, th_full + buf);
  };

  bool ok = true;
  int fetched = 0, landed = 0;   // parameter copies issued / waited for (leader)
  bool mma_pending = false;
  if (leader && (int)blockIdx.x < tiles) {
    fetch(blockIdx.x, 0);
    fetched = 1;
  }
  uint32_t mma_count = 0;
  int it = 0;
  // this thread's columns of its row: half `half` of the block's B columns
  constexpr int HC = B / 2;
  for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
    const int buf = it % Geo::NTH;
    const TileSide* sd;
    int b0, nbt;
    locate(t, sd, b0, nbt);
    bool lok = true;
    if (leader) {
      // two buffers: the next tile's parameters come in while this tile's
      // chain runs (the buffer was last read by the tile before this one,
      // finished below); one buffer: this tile's own, after the last one's
      const int next = Geo::NTH == 2 ? t + (int)gridDim.x : (it > 0 ? t : tiles);
      if (next < tiles) {
        fence_proxy_async_smem();   // generic reads of the buffer before the copy's writes
        fetch(next, Geo::NTH == 2 ? buf ^ 1 : 0);
        ++fetched;
      }
      lok = mbar_poll(th_full + buf, (uint32_t)(it / Geo::NTH) & 1, err);
      if (lok) ++landed;
    }
    if (__syncthreads_or(!lok)) {   // every thread leaves together
      ok = false;
      break;
    }
    const float* th = th_buf + buf * (Geo::th_bytes / 4) + g * P;
    const bool live = g < nbt;   // rows of a missing block (last tile) stay zero

    // ---- unpack: B = -K, A = X_1 = K on this row, columns of atom `half`
    // (block-diagonal: zeros outside the row's block)
#pragma unroll 1
    for (int k8 = half * 64; k8 < half * 64 + 64; k8 += 8) {
      uint32_t bh[4] = {0, 0, 0, 0}, bl[4] = {0, 0, 0, 0};
      if (live && k8 >= g * B && k8 < (g + 1) * B) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = -k_entry<B>(th, ri, k8 + e - g * B);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          if constexpr (F32) {
            uint32_t h0, l0, h1, l1;
            split_bf16(v[e], h0, l0);
            split_bf16(v[e + 1], h1, l1);
            bh[e / 2] = h0 | (h1 << 16);
            bl[e / 2] = l0 | (l1 << 16);
          } else {
            bh[e / 2] = bf16_bits(v[e]) | (bf16_bits(v[e + 1]) << 16);
          }
        }
      }
      const uint32_t off = op_off(r, k8);
      *reinterpret_cast<uint4*>(b_hi + off) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
      // bf16(-x) = -bf16(x): A = -B is a sign flip of every entry
      *reinterpret_cast<uint4*>(a_hi + off) =
          make_uint4(bh[0] ^ 0x80008000u, bh[1] ^ 0x80008000u, bh[2] ^ 0x80008000u,
                     bh[3] ^ 0x80008000u);
      if constexpr (F32) {
        *reinterpret_cast<uint4*>(b_lo + off) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
        *reinterpret_cast<uint4*>(a_lo + off) =
            make_uint4(bl[0] ^ 0x80008000u, bl[1] ^ 0x80008000u, bl[2] ^ 0x80008000u,
                       bl[3] ^ 0x80008000u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- the chain
    for (int i = 1; i <= n; ++i) {
      lok = true;
      if (leader) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 128, false, false);
        const uint32_t ah = smem_u32(a_hi), bhs = smem_u32(b_hi);
#pragma unroll
        for (int kc = 0; kc < 2; ++kc)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t o = kc * (128 * 128) + kk * 32;
            mma_bf16(tmem, sw128_desc(ah + o, 16, 1024), sw128_desc(bhs + o, 16, 1024), idesc,
                     (kc | kk) != 0);
            if constexpr (F32) {
              const uint32_t al = smem_u32(a_lo), bls = smem_u32(b_lo);
              mma_bf16(tmem, sw128_desc(ah + o, 16, 1024), sw128_desc(bls + o, 16, 1024), idesc, 1);
              mma_bf16(tmem, sw128_desc(al + o, 16, 1024), sw128_desc(bhs + o, 16, 1024), idesc, 1);
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
      for (int c0 = half * HC; c0 < (half + 1) * HC; c0 += (HC < 32 ? HC : 32)) {
        constexpr int W = HC < 32 ? HC : 32;   // columns per TMEM load
        uint32_t acc[W];
        const uint32_t ta = tmem + (uint32_t)(g * B + c0) + ((uint32_t)(quarter * 32) << 16);
        if constexpr (W == 32) tmem_ld32(ta, acc);
        else tmem_ld16(ta, acc);
        // 2K from the operand's own K (B = -K): bf16, or hi + lo for fp32 Q
        float k2[W];
#pragma unroll
        for (int q = 0; q < W / 8; ++q) {
          const uint32_t off = op_off(r, g * B + c0 + 8 * q);
          widen8(b_hi + off, k2 + 8 * q);
          if constexpr (F32) {
            float lo[8];
            widen8(b_lo + off, lo);
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
#pragma unroll
          for (int q = 0; q < W / 8; ++q) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              if constexpr (F32) {
                uint32_t h0, l0, h1, l1;
                split_bf16(x[8 * q + e], h0, l0);
                split_bf16(x[8 * q + e + 1], h1, l1);
                h[e / 2] = h0 | (h1 << 16);
                l[e / 2] = l0 | (l1 << 16);
              } else {
                h[e / 2] = bf16_bits(x[8 * q + e]) | (bf16_bits(x[8 * q + e + 1]) << 16);
              }
            }
            const uint32_t off = op_off(r, g * B + c0 + 8 * q);
            *reinterpret_cast<uint4*>(a_hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
            if constexpr (F32)
              *reinterpret_cast<uint4*>(a_lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
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
      if (i < n) fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();   // next operand written / this tile's parameters no longer read
    }
    if (!ok) break;
  }
  if (!ok && leader) {
    // wind-down after an expired wait: the copies and MMAs already issued
    // finish (bounded waits) before the CTA frees its memory
    for (int k = landed; k < fetched; ++k)
      mbar_wait_bounded(th_full + k % Geo::NTH, (uint32_t)(k / Geo::NTH) & 1, 1u << 16, nullptr);
    if (mma_pending) mbar_wait_bounded(mma_done, mma_count & 1, 1u << 16, nullptr);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int B, bool F32>
poetx_status tile_launch(const TileSide& s0, const TileSide& s1, int n, cudaStream_t s) {
  using Geo = TileGeo<B, F32>;
  const void* kern = (const void*)cnp_tile_kernel<B, F32>;
  if (set_max_dynamic_smem(kern, Geo::smem) != cudaSuccess) return check_launch();
  const int tiles = (s0.nb + Geo::G - 1) / Geo::G + (s1.nb + Geo::G - 1) / Geo::G;
  // CTAs resident per SM (shared memory and TMEM: 128 columns each)
  int per_sm = Geo::per_sm(Geo::smem);
  if (per_sm > 4) per_sm = 4;
  if (per_sm < 1) per_sm = 1;
  int grid = device_sm_count() * per_sm;
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
