// tc_cluster_apply.cu -- permuted block-diagonal apply across a thread-block cluster.
//
// [POET-X §2.B-§2.C] ("POET-X: Memory-efficient LLM Training by Scaling
// Orthogonal Transformation", gist.science summary, sections 2.B and 2.C):
// the orthogonal factors are block-diagonal (every b x b block its own small
// matrix, processed as a batch) and sandwiched between permutations applied
// as index maps.  For token t and block j this computes
//   GATHER_IN    out[t][j*b + i]       = sum_k Qop_j[i][k] in[t][perm[j*b + k]]
//   SCATTER_OUT  out[t][perm[j*b + i]] = sum_k Qop_j[i][k] in[t][j*b + k]
// with Qop_j = Q_j or Q_j^T (u = x_pi B_P^T and g_z = dy_pi B_R; y =
// scatter(z B_R^T) and dX = scatter(g_u B_P)).
//
// A cluster of C CTAs works on one 64-token tile at a time.  CTA c owns the
// natural feature columns [c*F, (c+1)*F) (F = d/C) for loading or storing, and
// the blocks [c*G, (c+1)*G) (G = d/(b*C)) for the products, whose Qop blocks
// it keeps in tensor memory for the whole launch (the MMA reads A from TMEM).
// The permutation is carried out on chip: 16-byte pieces (8 tokens of one
// feature) travel between the CTAs' shared memories with st.async, each
// counted against the receiving CTA's mbarrier, so no permuted copy of an
// activation is ever written to HBM and every activation byte crosses HBM
// once.
//   GATHER_IN:   TMA loads the tile's own columns [64 tokens x F] -> worker
//                warps cut them into feature pieces and send each to the CTA
//                that owns its block, at its gathered position -> that CTA's
//                MMA (M = 128 outputs, N = 64 tokens, K = 16) reads the
//                received [b features x 64 tokens] operand -> the epilogue
//                writes the block's contiguous output columns.
//   SCATTER_OUT: TMA loads the own blocks' contiguous input columns -> MMA ->
//                the epilogue sends each output feature (a TMEM lane) to the
//                CTA owning its scattered column -> that CTA transposes the
//                received [F features x 64 tokens] to token rows and stores
//                them with TMA.
// Flow control: a receive buffer is refilled only after its owner has
// released it to every sender (remote mbarrier arrive).  Every wait is
// bounded (see tc_ptx.cuh); the cluster barriers at start and end are
// reached by every thread unconditionally.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

constexpr int TT = 64;                 // tokens per tile (MMA N)
constexpr int kCaThreads = 448;        // warp 0 TMA, warp 1 MMA, warps 2..9 movers, 10..13 epilogue
constexpr int kMovers = 256;
constexpr int kSmemLimit = 232448;

struct CaGeo {
  int C, G, F;        // cluster size, blocks per CTA, features per CTA
  int NS, NR, NA;     // ring depths: staged input, receive buffers, accumulators
  int s_bytes, r_bytes, st_bytes;
  int q_cols, a_cols, tmem_cols;
  int hdr;            // barriers + routing table, in front of the pipeline buffers
  int smem;
};

__device__ __forceinline__ void movers_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kMovers) : "memory");
}

__device__ __forceinline__ uint4 pack8f(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Loads Qop_j of the CTA's G blocks into tensor memory (lanes = rows i, two
// bf16 of consecutive k per 32-bit column), staging Q through shared memory.
// Called by all threads; `stage` must hold G * B * B bf16.
template <int B>
__device__ void load_q_to_tmem(const __nv_bfloat16* __restrict__ Q, int j0, int G, int transpose_q,
                               uint8_t* stage, uint32_t tmem_base) {
  constexpr int P = B + 8;   // padded row pitch (elements): row reads of 16 bytes avoid conflicts
  const uint4* src = reinterpret_cast<const uint4*>(Q + (size_t)j0 * B * B);
  for (int u = threadIdx.x; u < G * B * B / 8; u += blockDim.x) {
    const int row = u / (B / 8), c8 = u % (B / 8);
    *reinterpret_cast<uint4*>(stage + ((size_t)row * P + c8 * 8) * 2) = __ldg(src + u);
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp >= 10) {
    const int quarter = warp % 4;
    const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(stage);
    constexpr int halves = B / 128;
    for (int jj = 0; jj < G; ++jj)
      for (int h = 0; h < halves; ++h) {
        const int i = h * 128 + quarter * 32 + lane;
        const __nv_bfloat16* blk = qs + (size_t)jj * B * P;
        const uint32_t col0 = (uint32_t)((jj * halves + h) * (B / 2));
        for (int c = 0; c < B / 2; c += 32) {
          uint32_t r[32];
          if (transpose_q) {
            // row i of Q^T is column i of Q: lanes read consecutive columns of one row
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int k = 2 * (c + e);
              r[e] = (uint32_t)__bfloat16_as_ushort(blk[(size_t)k * P + i]) |
                     ((uint32_t)__bfloat16_as_ushort(blk[(size_t)(k + 1) * P + i]) << 16);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 v = *reinterpret_cast<const uint4*>(blk + (size_t)i * P + 2 * c + 8 * q);
              r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
            }
          }
          tmem_st32(tmem_base + col0 + (uint32_t)c + ((uint32_t)(quarter * 32) << 16), r);
        }
      }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// ======================================================================== GATHER_IN
template <int B>
__global__ void __launch_bounds__(kCaThreads, 1)
    ca_gather_kernel(const __grid_constant__ CUtensorMap tmIn, const __nv_bfloat16* __restrict__ Q,
                     const int32_t* __restrict__ inv, __nv_bfloat16* __restrict__ out, int T, int d,
                     CaGeo g, int transpose_q, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  const int C = g.C, G = g.G, F = g.F;
  const int s_off = g.hdr;
  const int r_off = s_off + g.NS * g.s_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* s_full = bars;          // [2]
  uint64_t* s_empty = bars + 2;     // [2]
  uint64_t* r_full = bars + 4;      // [2]
  uint64_t* dst_free = bars + 6;    // [2]
  uint64_t* a_full = bars + 8;      // [2]
  uint64_t* a_empty = bars + 10;    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + 256);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int n_clusters = gridDim.x / C;
  const int n_tiles = (T + TT - 1) / TT;
  const int r_bytes = g.r_bytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_empty + i, kMovers);
      mbar_init(r_full + i, 1);
      mbar_init(dst_free + i, C);
      mbar_init(a_full + i, 1);
      mbar_init(a_empty + i, 128);
    }
    fence_mbar_init();
    // the first use of every receive buffer expects G blocks x b features x 64 tokens
    for (int i = 0; i < g.NR; ++i) mbar_arrive_expect_tx(r_full + i, (uint32_t)r_bytes);
  }
  if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)g.tmem_cols);
  // destination of each owned feature: (CTA << 24) | byte offset of its K row in the buffer
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    const int p = __ldg(inv + c * F + f);
    const int j = p / B, k = p % B;
    const int dest = j / G, jj = j % G;
    table[f] = ((uint32_t)dest << 24) |
               (uint32_t)(jj * (B * TT * 2) + (k >> 3) * 1024 + (k & 7) * 128);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  load_q_to_tmem<B>(Q, c * G, G, transpose_q, smem + g.hdr, tmem_base);
  cluster_sync();   // every CTA's barriers are initialised before any remote access

  const uint32_t acc0 = tmem_base + (uint32_t)g.q_cols;
  bool ok = true;
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        const int s = it % g.NS;
        if (!(ok = mbar_wait(s_empty + s, ((it / g.NS) & 1) ^ 1, err))) break;
        mbar_arrive_expect_tx(s_full + s, (uint32_t)g.s_bytes);
        uint8_t* dst = smem + s_off + s * g.s_bytes;
        for (int q = 0; q < F / 64; ++q)
          tma_load_2d(dst + q * (TT * 128), &tmIn, c * F + q * 64, tile * TT, s_full + s);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TT, false, true);
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        const int r = it % g.NR, a = it % g.NA;
        if (!(ok = mbar_wait_cluster(r_full + r, (it / g.NR) & 1, err))) break;
        mbar_arrive_expect_tx(r_full + r, (uint32_t)r_bytes);   // the buffer's next use
        fence_proxy_async_smem();
        if (!(ok = mbar_wait(a_empty + a, ((it / g.NA) & 1) ^ 1, err))) break;
        tc_fence_after();
        const uint32_t rb = smem_u32(smem + r_off + r * r_bytes);
        for (int jj = 0; jj < G; ++jj)
          for (int h = 0; h < halves; ++h) {
            const uint32_t d_tmem = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT);
            const uint32_t a_tmem = tmem_base + (uint32_t)((jj * halves + h) * (B / 2));
#pragma unroll 4
            for (int kk = 0; kk < B / 16; ++kk) {
              const uint64_t bdesc = sw128_desc(rb + jj * (B * TT * 2) + kk * 2048, B * 128, 1024);
              mma_bf16_ts(d_tmem, a_tmem + (uint32_t)(kk * 8), bdesc, idesc, kk != 0);
            }
          }
        mma_commit(a_full + a);
      }
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------------- movers: send feature pieces
    const int pt = threadIdx.x - 64;
    const uint32_t rbase = smem_u32(smem + r_off);
    const uint32_t rfull0 = smem_u32(r_full);
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int s = it % g.NS, r = it % g.NR;
      if (!(ok = mbar_wait(s_full + s, (it / g.NS) & 1, err))) break;
      if (!(ok = mbar_wait_cluster(dst_free + r, ((it / g.NR) & 1) ^ 1, err))) break;
      const uint8_t* S = smem + s_off + s * g.s_bytes;
      for (int w = pt; w < F * (TT / 8); w += kMovers) {
        const int f = w % F, grp = w / F, t8 = grp * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int row = t8 + e;
          const uint32_t off = (uint32_t)((f >> 6) * (TT * 128) + row * 128 +
                                          ((((f >> 3) & 7) ^ (row & 7)) << 4) + (f & 7) * 2);
          v[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(S + off));
        }
        const uint32_t ent = table[f];
        const uint32_t dest = ent >> 24, roff = ent & 0xFFFFFFu;
        const uint32_t k7 = (roff >> 7) & 7u;
        const uint32_t laddr = rbase + (uint32_t)(r * r_bytes) + roff + ((((uint32_t)grp) ^ k7) << 4);
        st_async_v4(mapa_shared(laddr, dest), pack8f(v), mapa_shared(rfull0 + 8u * r, dest));
      }
      mbar_arrive(s_empty + s);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp % 4;
    const uint32_t dfree0 = smem_u32(dst_free);
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int r = it % g.NR, a = it % g.NA;
      if (!(ok = mbar_wait(a_full + a, (it / g.NA) & 1, err))) break;
      tc_fence_after();
      if (warp == 10 && lane == 0)   // this tile's receive buffer has been read by the MMAs
        for (int q = 0; q < C; ++q) mbar_arrive_remote(mapa_shared(dfree0 + 8u * r, (uint32_t)q));
      const int t0 = tile * TT;
      for (int jj = 0; jj < G; ++jj)
        for (int h = 0; h < halves; ++h) {
          const int i = h * 128 + quarter * 32 + lane;
          __nv_bfloat16* o = out + (size_t)((c * G + jj) * B + i);
          const uint32_t tacc = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT) +
                                ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
          for (int cc = 0; cc < TT; cc += 32) {
            uint32_t rr[32];
            tmem_ld32(tacc + (uint32_t)cc, rr);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t0 + cc + t < T) o[(size_t)(t0 + cc + t) * d] = __float2bfloat16_rn(__uint_as_float(rr[t]));
          }
        }
      tc_fence_before();
      mbar_arrive(a_empty + a);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves while another may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)g.tmem_cols);
  }
}

// ======================================================================== SCATTER_OUT
template <int B>
__global__ void __launch_bounds__(kCaThreads, 1)
    ca_scatter_kernel(const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ CUtensorMap tmOut,
                      const __nv_bfloat16* __restrict__ Q, const int32_t* __restrict__ perm, int T,
                      int d, CaGeo g, int transpose_q, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  const int C = g.C, G = g.G, F = g.F;
  const int s_off = g.hdr;
  const int r_off = s_off + g.NS * g.s_bytes;
  const int st_off = r_off + g.NR * g.r_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* s_full = bars;          // [2] input tile landed
  uint64_t* s_empty = bars + 2;     // [2] input tile read by the MMAs
  uint64_t* r_full = bars + 4;      // [2] receive buffer complete (st.async bytes)
  uint64_t* dst_free = bars + 6;    // [2] every owner released its receive buffer
  uint64_t* a_full = bars + 8;      // [2]
  uint64_t* a_empty = bars + 10;    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + 256);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int n_clusters = gridDim.x / C;
  const int n_tiles = (T + TT - 1) / TT;
  const int r_bytes = g.r_bytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_empty + i, 1);
      mbar_init(r_full + i, 1);
      mbar_init(dst_free + i, C);
      mbar_init(a_full + i, 1);
      mbar_init(a_empty + i, 128);
    }
    fence_mbar_init();
    for (int i = 0; i < g.NR; ++i) mbar_arrive_expect_tx(r_full + i, (uint32_t)r_bytes);
  }
  if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)g.tmem_cols);
  // owner of each output feature of the own blocks: (CTA << 24) | byte offset of its row
  for (int e = threadIdx.x; e < G * B; e += blockDim.x) {
    const int nc = __ldg(perm + c * G * B + e);
    table[e] = ((uint32_t)(nc / F) << 24) | (uint32_t)((nc % F) * 128);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  load_q_to_tmem<B>(Q, c * G, G, transpose_q, smem + g.hdr, tmem_base);
  cluster_sync();

  const uint32_t acc0 = tmem_base + (uint32_t)g.q_cols;
  bool ok = true;
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: own blocks' columns
    if (lane == 0) {
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        const int s = it % g.NS;
        if (!(ok = mbar_wait(s_empty + s, ((it / g.NS) & 1) ^ 1, err))) break;
        mbar_arrive_expect_tx(s_full + s, (uint32_t)g.s_bytes);
        uint8_t* dst = smem + s_off + s * g.s_bytes;
        for (int jj = 0; jj < G; ++jj)
          for (int q = 0; q < B / 64; ++q)
            tma_load_2d(dst + jj * (TT * B * 2) + q * (TT * 128), &tmIn, (c * G + jj) * B + q * 64,
                        tile * TT, s_full + s);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TT, false, false);
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        const int s = it % g.NS, a = it % g.NA;
        if (!(ok = mbar_wait(s_full + s, (it / g.NS) & 1, err))) break;
        if (!(ok = mbar_wait(a_empty + a, ((it / g.NA) & 1) ^ 1, err))) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(smem + s_off + s * g.s_bytes);
        for (int jj = 0; jj < G; ++jj)
          for (int h = 0; h < halves; ++h) {
            const uint32_t d_tmem = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT);
            const uint32_t a_tmem = tmem_base + (uint32_t)((jj * halves + h) * (B / 2));
#pragma unroll 4
            for (int kk = 0; kk < B / 16; ++kk) {
              const uint64_t bdesc =
                  sw128_desc(sb + jj * (TT * B * 2) + (kk >> 2) * (TT * 128) + (kk & 3) * 32, 16, 1024);
              mma_bf16_ts(d_tmem, a_tmem + (uint32_t)(kk * 8), bdesc, idesc, kk != 0);
            }
          }
        mma_commit(s_empty + s);
        mma_commit(a_full + a);
      }
    }
  } else if (warp >= 10) {
    // ---------------------------------------------------------------- epilogue: send output features
    const int quarter = warp % 4;
    const uint32_t rbase = smem_u32(smem + r_off);
    const uint32_t rfull0 = smem_u32(r_full);
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int r = it % g.NR, a = it % g.NA;
      if (!(ok = mbar_wait(a_full + a, (it / g.NA) & 1, err))) break;
      if (!(ok = mbar_wait_cluster(dst_free + r, ((it / g.NR) & 1) ^ 1, err))) break;
      tc_fence_after();
      for (int jj = 0; jj < G; ++jj)
        for (int h = 0; h < halves; ++h) {
          const int i = h * 128 + quarter * 32 + lane;
          const uint32_t ent = table[jj * B + i];
          const uint32_t owner = ent >> 24, roff = ent & 0xFFFFFFu;
          const uint32_t f7 = (roff >> 7) & 7u;
          const uint32_t laddr = rbase + (uint32_t)(r * r_bytes) + roff;
          const uint32_t raddr = mapa_shared(laddr, owner);
          const uint32_t rbar = mapa_shared(rfull0 + 8u * r, owner);
          const uint32_t tacc = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT) +
                                ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
          for (int cc = 0; cc < TT; cc += 32) {
            uint32_t rr[32];
            tmem_ld32(tacc + (uint32_t)cc, rr);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t grp = (uint32_t)(cc / 8 + u);
              const uint4 v = make_uint4(
                  pack_bf16x2(__uint_as_float(rr[8 * u + 0]), __uint_as_float(rr[8 * u + 1])),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 2]), __uint_as_float(rr[8 * u + 3])),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 4]), __uint_as_float(rr[8 * u + 5])),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 6]), __uint_as_float(rr[8 * u + 7])));
              st_async_v4(raddr + ((grp ^ f7) << 4), v, rbar);
            }
          }
        }
      tc_fence_before();
      mbar_arrive(a_empty + a);
    }
  } else {
    // ---------------------------------------------------------------- movers: received features -> token rows
    const int pt = threadIdx.x - 64;
    const uint32_t dfree0 = smem_u32(dst_free);
    uint8_t* ST = smem + st_off;
    bool pending = false;
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int r = it % g.NR;
      if (!(ok = mbar_wait_cluster(r_full + r, (it / g.NR) & 1, err))) break;
      if (pt == 0) {
        mbar_arrive_expect_tx(r_full + r, (uint32_t)r_bytes);   // the buffer's next use
        if (pending) bulk_wait_read0();                        // the staging tile is free again
      }
      movers_bar();
      const uint8_t* R = smem + r_off + r * r_bytes;
      for (int w = pt; w < TT * (F / 8); w += kMovers) {
        const int t = w % TT, f8 = (w / TT) * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int fr = f8 + e;
          const uint32_t off = (uint32_t)(fr * 128 + ((((t >> 3) ^ (fr & 7)) & 7) << 4) + (t & 7) * 2);
          v[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(R + off));
        }
        const uint32_t so = (uint32_t)((f8 >> 6) * (TT * 128) + t * 128 +
                                       ((((f8 & 63) >> 3) ^ (t & 7)) << 4));
        *reinterpret_cast<uint4*>(ST + so) = pack8f(v);
      }
      fence_proxy_async_smem();
      movers_bar();
      if (pt == 0) {
        for (int q = 0; q < C; ++q) mbar_arrive_remote(mapa_shared(dfree0 + 8u * r, (uint32_t)q));
        for (int q = 0; q < F / 64; ++q) tma_store_2d(&tmOut, ST + q * (TT * 128), c * F + q * 64, tile * TT);
        bulk_commit();
        pending = true;
      }
    }
    if (pt == 0 && pending) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)g.tmem_cols);
  }
}

int tmem_alloc_cols(int used) {
  int c = 32;
  while (c < used) c *= 2;
  return c;
}

// Picks the cluster geometry for (d, b); returns false if none fits.  Cluster
// sizes up to 8 (portable) are preferred, then 9..16.
bool ca_geometry(int d, int b, bool gather, CaGeo* out) {
  if ((b != 128 && b != 256) || d % b) return false;
  const int nb = d / b;
  const int halves = b / 128;
  const int order[15] = {8, 7, 6, 5, 4, 3, 2, 16, 15, 14, 13, 12, 11, 10, 9};
  for (int oi = 0; oi < 15; ++oi) {
    const int C = order[oi];
    if (nb % C) continue;
    CaGeo g;
    g.C = C;
    g.G = nb / C;
    g.F = d / C;
    if (g.F % 64) continue;
    g.q_cols = g.G * halves * (b / 2);
    g.NA = 2;
    g.a_cols = 2 * g.G * halves * TT;
    if (g.q_cols + g.a_cols > 512) {
      g.NA = 1;
      g.a_cols = g.G * halves * TT;
    }
    if (g.q_cols + g.a_cols > 512) continue;
    g.tmem_cols = tmem_alloc_cols(g.q_cols + g.a_cols);
    if (gather) {
      g.s_bytes = TT * g.F * 2;            // own columns of the tile
      g.r_bytes = g.G * b * TT * 2;        // received operand of the own blocks
      g.st_bytes = 0;
    } else {
      g.s_bytes = g.G * TT * b * 2;        // own blocks' input columns
      g.r_bytes = g.F * TT * 2;            // received output features
      g.st_bytes = TT * g.F * 2;           // token-row staging for the TMA store
    }
    const int table = 4 * (gather ? g.F : g.G * b);
    g.hdr = (256 + table + 1023) / 1024 * 1024;
    const int qstage = g.G * b * (b + 8) * 2;
    bool found = false;
    for (int NS = 2; NS >= 1 && !found; --NS)
      for (int NR = 2; NR >= 1 && !found; --NR) {
        const int body = NS * g.s_bytes + NR * g.r_bytes + g.st_bytes;
        const int smem = 1024 + g.hdr + (body > qstage ? body : qstage);
        if (smem <= kSmemLimit) {
          g.NS = NS;
          g.NR = NR;
          g.smem = smem;
          found = true;
        }
      }
    if (!found) continue;
    *out = g;
    return true;
  }
  return false;
}

}  // namespace

bool cluster_apply_supported(int d, int b, bool scatter) {
  CaGeo g;
  return ca_geometry(d, b, !scatter, &g);
}

poetx_status cluster_apply_bf16(const void* in, void* out, const void* Q, const int32_t* perm,
                                const int32_t* inv, int T, int d, int b, bool transpose_q,
                                bool scatter, cudaStream_t s) {
  if (T <= 0) return POETX_OK;
  CaGeo g;
  if (!ca_geometry(d, b, !scatter, &g)) return POETX_ERR_UNSUPPORTED;
  CUtensorMap tin, tout;
  if (!make_tmap_2d(&tin, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, TT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  if (scatter && !make_tmap_2d(&tout, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T,
                               (uint64_t)d, TT, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  const void* kern;
  if (scatter)
    kern = b == 256 ? (const void*)ca_scatter_kernel<256> : (const void*)ca_scatter_kernel<128>;
  else
    kern = b == 256 ? (const void*)ca_gather_kernel<256> : (const void*)ca_gather_kernel<128>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem) != cudaSuccess)
    return check_launch();
  if (g.C > 8 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return check_launch();
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kCaThreads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once (persistent), but no more than tiles
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cfg.gridDim = dim3((sms / g.C) * g.C);
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess || active < 1) {
    cudaGetLastError();
    return POETX_ERR_UNSUPPORTED;
  }
  const int n_tiles = (T + TT - 1) / TT;
  const int clusters = active < n_tiles ? active : n_tiles;
  cfg.gridDim = dim3(clusters * g.C);
  int* err = device_error_word();
  const int tq = transpose_q ? 1 : 0;
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(Q);
  {
    KernelScope ks_(scatter ? "tc_cluster_scatter" : "tc_cluster_gather", s);
    cudaError_t e;
    if (scatter) {
      if (b == 256)
        e = cudaLaunchKernelEx(&cfg, ca_scatter_kernel<256>, tin, tout, qp, perm, T, d, g, tq, err);
      else
        e = cudaLaunchKernelEx(&cfg, ca_scatter_kernel<128>, tin, tout, qp, perm, T, d, g, tq, err);
    } else {
      __nv_bfloat16* op = static_cast<__nv_bfloat16*>(out);
      if (b == 256)
        e = cudaLaunchKernelEx(&cfg, ca_gather_kernel<256>, tin, qp, inv, op, T, d, g, tq, err);
      else
        e = cudaLaunchKernelEx(&cfg, ca_gather_kernel<128>, tin, qp, inv, op, T, d, g, tq, err);
    }
    if (e != cudaSuccess) return check_launch();
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
