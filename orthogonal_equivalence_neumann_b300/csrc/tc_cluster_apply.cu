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
// natural feature columns [c*F, (c+1)*F) (F = d/C) for loading or storing,
// and the blocks [c*G, (c+1)*G) (G = d/(b*C)) for the products, whose Qop it
// keeps in tensor memory for the whole launch (the MMA reads A from TMEM).
// Activations cross HBM once.  The permutation is carried out in 128-byte
// feature rows (the 64 tokens of one feature): a CTA writes each row it
// produces straight to its place in a small per-cluster exchange ring in the
// workspace (a few MB, rewritten every few microseconds, so it lives in L2),
// and the CTA that needs the rows fetches its whole part with one bulk copy.
// Hand-offs use cluster mbarriers (remote arrive after a cluster-scope fence).
//   GATHER_IN:   TMA loads the tile's own columns [64 tokens x F] -> mover
//                warps write each feature row to the part of the CTA owning
//                its block, at its gathered position -> that CTA's loader
//                fetches its [G*b features x 64 tokens] operand -> MMA
//                (M = 128 outputs, N = 64 tokens, K = 16) -> the epilogue
//                stages the output tile in token rows and stores it by TMA.
//   SCATTER_OUT: TMA loads the own blocks' contiguous input columns -> MMA ->
//                the epilogue writes each output feature row (a TMEM lane)
//                to the part of the CTA owning its scattered column -> that
//                CTA's loader fetches its [F features x 64 tokens] -> mover
//                warps transpose it to token rows -> TMA store.
// Flow control: a slot is rewritten only after every CTA that reads it has
// fetched it.  Every wait is bounded (see tc_ptx.cuh); the cluster barriers
// at start and end are reached by every thread unconditionally.
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_exchange.cuh"
#include "tc_ptx.cuh"
#include "tc_qstage.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

using namespace xchg;

constexpr int kCaThreads = 512;        // warp 0 TMA, 1 MMA, 2..9 movers, 10..13 epilogue, 14 loader, 15 signals
constexpr int kSmemLimit = 232448;
constexpr int kOneCtaSmem = 120 * 1024;

struct CaGeo {
  int C, G, F;        // cluster size, blocks per CTA, features per CTA
  int NS, NR, NA;     // ring depths: staged input, fetched parts in shared memory, accumulators
  int NST;            // output staging tiles (TMA store sources)
  int NX;             // exchange slots in the workspace ring
  int s_bytes;        // input tile in shared memory
  int r_bytes;        // one CTA's part of an exchange slot (rows of 128 bytes)
  int st_bytes;       // token-row staging of the output tile for the TMA store
  int q_cols, a_cols, tmem_cols;
  int hdr;            // barriers + routing table, in front of the pipeline buffers
  int q_rel;          // Q staging area, from the start of the pipeline buffers
  int smem;
};

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

// ======================================================================== GATHER_IN
template <int B>
__global__ void __launch_bounds__(kCaThreads, 1)
    ca_gather_kernel(const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ CUtensorMap tmOut,
                     const __grid_constant__ CUtensorMap tmQ, const int32_t* __restrict__ inv,
                     uint8_t* __restrict__ xchg, int T, CaGeo g, int transpose_q, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  const int C = g.C, G = g.G, F = g.F;
  const int s_off = g.hdr;
  const int r_off = s_off + g.NS * g.s_bytes;
  const int o_off = r_off + g.NR * g.r_bytes;
  const Bars br = bars_at(smem);
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + kTableOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int n_clusters = gridDim.x / C;
  const int n_tiles = (T + TT - 1) / TT;
  // exchange ring of this cluster: [slot r][reader CTA q][r_bytes]
  const int n_it = cluster_iters(cluster_id, n_clusters, n_tiles);
  const size_t slot_stride = (size_t)C * g.r_bytes;
  uint8_t* ring = xchg + (size_t)cluster_id * g.NX * slot_stride;

  if (threadIdx.x == 0) init_bars(br, C, kMovers, 1, kMovers);
  if (warp == 1) tmem_alloc(br.tmem_slot, (uint32_t)g.tmem_cols);
  gather_table<B>(table, inv, c, F, G);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *br.tmem_slot;
  // Q into tensor memory through a staging area of the pipeline buffers: at
  // their end when that leaves the input tiles free (q_rel > 0: the first
  // tiles load and move through the exchange while Q is staged; the loader
  // and the MMA wait for q_done), else at their start, before the first tiles
  const bool early = g.q_rel > 0;
  uint8_t* qst = smem + s_off + g.q_rel;
  if (threadIdx.x == 0) issue_q_loads(&tmQ, qst, c * G, G, B, br.q_full);
  bool ok = true;
  auto stage_q = [&]() {
    if (warp >= 10 && warp < 14) {
      if ((ok = mbar_wait(br.q_full, 0, err)))
        q_stage_to_tmem<B>(qst, G, transpose_q, tmem_base, warp % 4, lane);
      tc_fence_before();
      mbar_arrive(br.q_done);
    }
  };
  if (!early) {
    stage_q();
    tc_fence_before();
    __syncthreads();
  }
  // the first input tiles (disjoint from the staging area, or after it was read)
  int prefetched = 0;
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();
    for (int tile = cluster_id; tile < n_tiles && prefetched < g.NS; tile += n_clusters, ++prefetched) {
      mbar_arrive_expect_tx(br.s_full + prefetched, (uint32_t)g.s_bytes);
      uint8_t* dst = smem + s_off + prefetched * g.s_bytes;
      for (int q = 0; q < F / 64; ++q)
        tma_load_2d(dst + q * (TT * 128), &tmIn, c * F + q * 64, tile * TT, br.s_full + prefetched);
    }
  }
  cluster_sync();   // every CTA's barriers are initialised before any remote access
  tc_fence_after();
  if (early) stage_q();

  const uint32_t acc0 = tmem_base + (uint32_t)g.q_cols;
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: own columns of the tile
    if (lane == 0) {
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        if (it < prefetched) continue;
        const int s = it % g.NS;
        if (!(ok = mbar_wait(br.s_empty + s, ((it / g.NS) & 1) ^ 1, err))) break;
        mbar_arrive_expect_tx(br.s_full + s, (uint32_t)g.s_bytes);
        uint8_t* dst = smem + s_off + s * g.s_bytes;
        for (int q = 0; q < F / 64; ++q)
          tma_load_2d(dst + q * (TT * 128), &tmIn, c * F + q * 64, tile * TT, br.s_full + s);
      }
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------------- loader
    if (lane == 0)
      loader_loop(br, g.NR, g.NX, g.r_bytes, smem + r_off, ring + (size_t)c * g.r_bytes, slot_stride,
                  cluster_iters(cluster_id, n_clusters, n_tiles), ok, err, br.q_done);
  } else if (warp == 15) {
    // ---------------------------------------------------------------- signals to the readers
    signal_loop(br, g.NX, cluster_iters(cluster_id, n_clusters, n_tiles), C, lane, ok, err);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // The whole warp follows the fetched parts; lanes 1..C tell the writers
    // that this CTA's part of the slot has been fetched, lane 0 issues the MMAs.
    const uint32_t idesc = idesc_bf16(128, TT, false, true);
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int r = it % g.NR, a = it % g.NA;
      if (!(ok = mbar_wait(br.r_full + r, (it / g.NR) & 1, err))) break;
      if (lane >= 1) ack_fetch(br, it, g.NX, n_it, lane - 1, C);
      if (lane == 0) {
        if (it == 0 && !(ok = mbar_wait(br.q_done, 0, err))) break;   // Q is in tensor memory
        if (!(ok = mbar_wait(br.a_empty + a, ((it / g.NA) & 1) ^ 1, err))) break;
        tc_fence_after();
        const uint32_t rb = smem_u32(smem + r_off + r * g.r_bytes);
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
        mma_commit(br.r_empty + r);
        mma_commit(br.a_full + a);
      }
    }
  } else if (warp < 10) {
    // ---------------------------------------------------------------- movers: write feature rows
    // A mover owns features of the tile: it collects the 64 tokens of a
    // feature (8 x 16 bytes, placed in the row's 128-byte swizzle order) and
    // writes the row into the exchange part of the CTA owning its block.
    const int pt = threadIdx.x - 64;
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int s = it % g.NS, x = it % g.NX;
      if (!(ok = mbar_wait(br.s_full + s, (it / g.NS) & 1, err))) break;
      // every reader has fetched this slot's previous contents
      if (!(ok = mbar_wait_cluster(br.x_free + x, ((it / g.NX) & 1) ^ 1, err))) break;
      move_gather_rows(smem + s_off + s * g.s_bytes, ring + (size_t)x * slot_stride, table, F,
                       g.r_bytes, pt);
      mbar_arrive(br.s_empty + s);
      mbar_arrive(br.moved + x);   // the loader warp signals the readers
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // TMEM lanes are output features, columns tokens: each thread writes its
    // feature's 64 tokens into a token-row staging tile (128-byte swizzle, the
    // TMA store layout); one thread then stores the tile with TMA.
    const int quarter = warp % 4;
    const int et = threadIdx.x - 320;   // 0..127
    bool pending = false;
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int a = it % g.NA;
      uint8_t* ostg = smem + o_off + (it % g.NST) * g.st_bytes;
      if (!(ok = mbar_wait(br.a_full + a, (it / g.NA) & 1, err))) break;
      tc_fence_after();
      if (pending) {   // the store that last used this staging tile has finished reading it
        if (et == 0) {
          if (g.NST > 1) bulk_wait_read1();
          else bulk_wait_read0();
        }
        epi_bar();
      }
      for (int jj = 0; jj < G; ++jj)
        for (int h = 0; h < halves; ++h) {
          const int f = jj * B + h * 128 + quarter * 32 + lane;   // column within the CTA's blocks
          uint8_t* col = ostg + (f >> 6) * (TT * 128) + (f & 7) * 2;
          const uint32_t fu = (uint32_t)((f & 63) >> 3);
          const uint32_t tacc = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT) +
                                ((uint32_t)(quarter * 32) << 16);
          // both 32-token halves in flight before one wait
          uint32_t rr[2][32];
          tmem_ld32(tacc, rr[0]);
          tmem_ld32(tacc + 32u, rr[1]);
          tmem_ld_wait();
          tmem_regs_ready(rr[0]);
          tmem_regs_ready(rr[1]);
#pragma unroll
          for (int tr = 0; tr < TT; ++tr)
            *reinterpret_cast<__nv_bfloat16*>(col + tr * 128 + ((fu ^ (uint32_t)(tr & 7)) << 4)) =
                __float2bfloat16_rn(__uint_as_float(rr[tr >> 5][tr & 31]));
        }
      tc_fence_before();
      mbar_arrive(br.a_empty + a);   // the accumulators may be refilled
      fence_proxy_async_smem();
      epi_bar();
      if (et == 0) {
        for (int q = 0; q < G * B / 64; ++q)
          tma_store_2d(&tmOut, ostg + q * (TT * 128), c * G * B + q * 64, tile * TT);
        bulk_commit();
      }
      pending = true;
    }
    if (et == 0 && pending) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves before its cluster is done with the exchange
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)g.tmem_cols);
  }
}

// ======================================================================== SCATTER_OUT
template <int B>
__global__ void __launch_bounds__(kCaThreads, 1)
    ca_scatter_kernel(const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ CUtensorMap tmOut,
                      const __grid_constant__ CUtensorMap tmQ, const int32_t* __restrict__ perm,
                      uint8_t* __restrict__ xchg, int T, CaGeo g, int transpose_q, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  const int C = g.C, G = g.G, F = g.F;
  const int s_off = g.hdr;
  const int r_off = s_off + g.NS * g.s_bytes;
  const int st_off = r_off + g.NR * g.r_bytes;
  const Bars br = bars_at(smem);
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + kTableOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int n_clusters = gridDim.x / C;
  const int n_tiles = (T + TT - 1) / TT;
  const int n_it = cluster_iters(cluster_id, n_clusters, n_tiles);
  const size_t slot_stride = (size_t)C * g.r_bytes;
  uint8_t* ring = xchg + (size_t)cluster_id * g.NX * slot_stride;

  if (threadIdx.x == 0) init_bars(br, C, 1, 1, 128);
  if (warp == 1) tmem_alloc(br.tmem_slot, (uint32_t)g.tmem_cols);
  // each output feature of the own blocks: (owner CTA << 24) | byte offset of its row there
  for (int e = threadIdx.x; e < G * B; e += blockDim.x) {
    const int nc = __ldg(perm + c * G * B + e);
    table[e] = ((uint32_t)(nc / F) << 24) | (uint32_t)((nc % F) * 128);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *br.tmem_slot;
  // Q into tensor memory through a staging area of the pipeline buffers: at
  // their end when that leaves the input tiles free (q_rel > 0: the first
  // tiles load and move through the exchange while Q is staged; the loader
  // and the MMA wait for q_done), else at their start, before the first tiles
  const bool early = g.q_rel > 0;
  uint8_t* qst = smem + s_off + g.q_rel;
  if (threadIdx.x == 0) issue_q_loads(&tmQ, qst, c * G, G, B, br.q_full);
  bool ok = true;
  auto stage_q = [&]() {
    if (warp >= 10 && warp < 14) {
      if ((ok = mbar_wait(br.q_full, 0, err)))
        q_stage_to_tmem<B>(qst, G, transpose_q, tmem_base, warp % 4, lane);
      tc_fence_before();
      mbar_arrive(br.q_done);
    }
  };
  if (!early) {
    stage_q();
    tc_fence_before();
    __syncthreads();
  }
  // the first input tiles (disjoint from the staging area, or after it was read)
  int prefetched = 0;
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();
    for (int tile = cluster_id; tile < n_tiles && prefetched < g.NS; tile += n_clusters, ++prefetched) {
      mbar_arrive_expect_tx(br.s_full + prefetched, (uint32_t)g.s_bytes);
      uint8_t* dst = smem + s_off + prefetched * g.s_bytes;
      for (int jj = 0; jj < G; ++jj)
        for (int q = 0; q < B / 64; ++q)
          tma_load_2d(dst + jj * (TT * B * 2) + q * (TT * 128), &tmIn, (c * G + jj) * B + q * 64,
                      tile * TT, br.s_full + prefetched);
    }
  }
  cluster_sync();   // every CTA's barriers are initialised before any remote access
  tc_fence_after();
  if (early) stage_q();

  const uint32_t acc0 = tmem_base + (uint32_t)g.q_cols;
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA: own blocks' columns
    if (lane == 0) {
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        if (it < prefetched) continue;
        const int s = it % g.NS;
        if (!(ok = mbar_wait(br.s_empty + s, ((it / g.NS) & 1) ^ 1, err))) break;
        mbar_arrive_expect_tx(br.s_full + s, (uint32_t)g.s_bytes);
        uint8_t* dst = smem + s_off + s * g.s_bytes;
        for (int jj = 0; jj < G; ++jj)
          for (int q = 0; q < B / 64; ++q)
            tma_load_2d(dst + jj * (TT * B * 2) + q * (TT * 128), &tmIn, (c * G + jj) * B + q * 64,
                        tile * TT, br.s_full + s);
      }
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------------- loader
    if (lane == 0)
      loader_loop(br, g.NR, g.NX, g.r_bytes, smem + r_off, ring + (size_t)c * g.r_bytes, slot_stride,
                  cluster_iters(cluster_id, n_clusters, n_tiles), ok, err, br.q_done);
  } else if (warp == 15) {
    // ---------------------------------------------------------------- signals to the readers
    signal_loop(br, g.NX, cluster_iters(cluster_id, n_clusters, n_tiles), C, lane, ok, err);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TT, false, false);
      for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
        const int s = it % g.NS, a = it % g.NA;
        if (it == 0 && !(ok = mbar_wait(br.q_done, 0, err))) break;   // Q is in tensor memory
        if (!(ok = mbar_wait(br.s_full + s, (it / g.NS) & 1, err))) break;
        if (!(ok = mbar_wait(br.a_empty + a, ((it / g.NA) & 1) ^ 1, err))) break;
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
        mma_commit(br.s_empty + s);
        mma_commit(br.a_full + a);
      }
    }
  } else if (warp >= 10) {
    // ---------------------------------------------------------------- epilogue: write output feature rows
    // A thread owns one output feature (its TMEM lane): its 64 tokens become a
    // 128-byte row (8 x 16 bytes in the row's swizzle order), written into the
    // exchange part of the CTA owning the feature's scattered column.
    const int quarter = warp % 4;
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int x = it % g.NX, a = it % g.NA;
      if (!(ok = mbar_wait(br.a_full + a, (it / g.NA) & 1, err))) break;
      if (!(ok = mbar_wait_cluster(br.x_free + x, ((it / g.NX) & 1) ^ 1, err))) break;
      tc_fence_after();
      uint8_t* slot = ring + (size_t)x * slot_stride;
      for (int jj = 0; jj < G; ++jj)
        for (int h = 0; h < halves; ++h) {
          const int i = h * 128 + quarter * 32 + lane;
          const uint32_t ent = table[jj * B + i];
          const uint32_t roff = ent & 0xFFFFFFu;
          const uint32_t f7 = (roff >> 7) & 7u;
          uint8_t* row = slot + (size_t)(ent >> 24) * g.r_bytes + roff;
          const uint32_t tacc = acc0 + (uint32_t)(((a * G + jj) * halves + h) * TT) +
                                ((uint32_t)(quarter * 32) << 16);
          // both 32-token halves in flight before one wait
          uint32_t rr[2][32];
          tmem_ld32(tacc, rr[0]);
          tmem_ld32(tacc + 32u, rr[1]);
          tmem_ld_wait();
          tmem_regs_ready(rr[0]);
          tmem_regs_ready(rr[1]);
#pragma unroll
          for (int grp = 0; grp < TT / 8; ++grp) {
            const uint32_t* q = &rr[grp >> 2][(grp & 3) * 8];
            const uint4 v = make_uint4(pack_bf16x2(__uint_as_float(q[0]), __uint_as_float(q[1])),
                                       pack_bf16x2(__uint_as_float(q[2]), __uint_as_float(q[3])),
                                       pack_bf16x2(__uint_as_float(q[4]), __uint_as_float(q[5])),
                                       pack_bf16x2(__uint_as_float(q[6]), __uint_as_float(q[7])));
            *reinterpret_cast<uint4*>(row + ((((uint32_t)grp) ^ f7) << 4)) = v;
          }
        }
      tc_fence_before();
      mbar_arrive(br.a_empty + a);
      mbar_arrive(br.moved + x);   // the loader warp signals the readers
    }
  } else {
    // ---------------------------------------------------------------- movers: fetched features -> token rows
    const int pt = threadIdx.x - 64;
    bool pending = false;
    for (int it = 0, tile = cluster_id; tile < n_tiles && ok; tile += n_clusters, ++it) {
      const int r = it % g.NR;
      uint8_t* ST = smem + st_off + (it % g.NST) * g.st_bytes;
      if (!(ok = mbar_wait(br.r_full + r, (it / g.NR) & 1, err))) break;
      ack_fetch(br, it, g.NX, n_it, pt, C);   // this CTA's part has been fetched
      if (pt == 0 && pending) {   // the store that last used this staging tile has read it
        if (g.NST > 1) bulk_wait_read1();
        else bulk_wait_read0();
      }
      movers_bar();
      const uint8_t* R = smem + r_off + r * g.r_bytes;
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
        mbar_arrive(br.r_empty + r);            // the fetched part has been read
        for (int q = 0; q < F / 64; ++q) tma_store_2d(&tmOut, ST + q * (TT * 128), c * F + q * 64, tile * TT);
        bulk_commit();
        pending = true;
      }
    }
    if (pt == 0 && pending) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves before its cluster is done with the exchange
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
// sizes up to 8 (portable) only: larger clusters fit one per GPC, and at the
// 2048 -> 5632 layer (44 blocks of 128: 11-CTA clusters) the column
// permutation plus the unpermuted apply measured faster (1.13 vs 1.40 ms per
// training step).
bool ca_geometry(int d, int b, bool gather, CaGeo* out) {
  if ((b != 128 && b != 256) || d % b) return false;
  const int nb = d / b;
  const int halves = b / 128;
  const int order[7] = {8, 7, 6, 5, 4, 3, 2};
  for (int oi = 0; oi < 7; ++oi) {
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
      g.r_bytes = g.G * b * TT * 2;        // fetched operand of the own blocks
      g.st_bytes = g.G * b * TT * 2;       // output tile of the own blocks, token rows
    } else {
      g.s_bytes = g.G * TT * b * 2;        // own blocks' input columns
      g.r_bytes = g.F * TT * 2;            // fetched output features
      g.st_bytes = TT * g.F * 2;           // token-row staging for the TMA store
    }
    const int table = 4 * (gather ? g.F : g.G * b);
    g.hdr = (kTableOff + table + 1023) / 1024 * 1024;
    const int qstage = g.G * b * b * 2;   // staged in the pipeline buffers before first use
    // three fetched parts first (the exchange hand-off is the longest wait;
    // measured best at the square 2048 layer), then deeper input rings (they
    // hide the HBM latency), then double output staging (the TMA store of one
    // tile overlaps the next)
    const int cand[9][3] = {{2, 2, 3}, {4, 2, 2}, {3, 2, 2}, {4, 1, 2}, {3, 1, 2},
                            {2, 2, 2}, {2, 1, 2}, {2, 1, 1}, {1, 1, 1}};
    bool found = false;
    for (int ci = 0; ci < 9 && !found; ++ci) {
      const int NS = cand[ci][0], NST = cand[ci][1], NR = cand[ci][2];
      const int body = NS * g.s_bytes + NR * g.r_bytes + NST * g.st_bytes;
      const int smem = 1024 + g.hdr + body;
      if (smem <= kSmemLimit && qstage <= body) {
        g.NS = NS;
        g.NR = NR;
        g.NST = NST;
        // Q staged at the end of the buffers when that leaves the input tiles
        // free (the first tiles then load while Q goes to tensor memory)
        g.q_rel = body - qstage >= NS * g.s_bytes ? body - qstage : 0;
        // at most one CTA per SM, so a CTA never waits for another's tensor memory
        g.smem = smem > kOneCtaSmem ? smem : kOneCtaSmem;
        found = true;
      }
    }
    if (!found) continue;
    g.NX = kMaxSlots;
    *out = g;
    return true;
  }
  return false;
}

const void* ca_kernel_ptr(int b, bool scatter) {
  if (scatter) return b == 256 ? (const void*)ca_scatter_kernel<256> : (const void*)ca_scatter_kernel<128>;
  return b == 256 ? (const void*)ca_gather_kernel<256> : (const void*)ca_gather_kernel<128>;
}

// Clusters of one launch over T tokens (as many as fit at once, at most one per
// tile) and the exchange slots of each; false if the kernel cannot be resident.
bool ca_plan(int T, int b, bool scatter, CaGeo* g, int* clusters) {
  const void* kern = ca_kernel_ptr(b, scatter);
  if (set_max_dynamic_smem(kern, g->smem) != cudaSuccess ||
      (g->C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kCaThreads);
  cfg.dynamicSmemBytes = g->smem;
  const int sms = device_sm_count();
  cfg.gridDim = dim3((sms / g->C) * g->C);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g->C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = max_active_clusters(kern, cfg);
  if (n > sms / g->C) n = sms / g->C;
  const int n_tiles = (T + TT - 1) / TT;
  if (n > n_tiles) n = n_tiles;
  if (n < 1) return false;
  *clusters = n;
  g->NX = ring_slots(n_tiles, n);
  return true;
}

}  // namespace

bool cluster_apply_supported(int d, int b, bool scatter) {
  CaGeo g;
  return ca_geometry(d, b, !scatter, &g);
}

// Clusters of a launch over T tokens (0 if the cluster form does not apply).
int cluster_apply_clusters(int T, int d, int b, bool scatter) {
  CaGeo g;
  int clusters = 0;
  if (T <= 0 || !ca_geometry(d, b, !scatter, &g) || !ca_plan(T, b, scatter, &g, &clusters)) return 0;
  return clusters;
}

// Exchange ring: NX slots of C parts for each cluster of the launch.
size_t cluster_apply_workspace_bytes(int T, int d, int b, bool scatter) {
  CaGeo g;
  int clusters = 0;
  if (T <= 0 || !ca_geometry(d, b, !scatter, &g) || !ca_plan(T, b, scatter, &g, &clusters)) return 0;
  return (size_t)clusters * g.NX * g.C * g.r_bytes;
}

poetx_status cluster_apply_bf16(const void* in, void* out, const void* Q, const int32_t* perm,
                                const int32_t* inv, int T, int d, int b, bool transpose_q,
                                bool scatter, void* ws, size_t ws_bytes, cudaStream_t s, int max_clusters) {
  if (T <= 0) return POETX_OK;
  CaGeo g;
  if (!ca_geometry(d, b, !scatter, &g)) return POETX_ERR_UNSUPPORTED;
  int clusters = 0;
  if (!ca_plan(T, b, scatter, &g, &clusters)) return POETX_ERR_UNSUPPORTED;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  if (!ws || ws_bytes < (size_t)clusters * g.NX * g.C * g.r_bytes ||
      (reinterpret_cast<uintptr_t>(ws) & 255))
    return POETX_ERR_SHAPE;
  CUtensorMap tin, tout, tq;
  if (!make_tmap_2d(&tin, in, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, TT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tout, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, TT,
                    64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tq, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)b, 64, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * g.C);
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
  int* err = device_error_word();
  const int tqf = transpose_q ? 1 : 0;
  uint8_t* xchg = static_cast<uint8_t*>(ws);
  {
    KernelScope ks_(scatter ? "tc_cluster_scatter" : "tc_cluster_gather", s);
    cudaError_t e;
    if (scatter) {
      if (b == 256)
        e = cudaLaunchKernelEx(&cfg, ca_scatter_kernel<256>, tin, tout, tq, perm, xchg, T, g, tqf, err);
      else
        e = cudaLaunchKernelEx(&cfg, ca_scatter_kernel<128>, tin, tout, tq, perm, xchg, T, g, tqf, err);
    } else {
      if (b == 256)
        e = cudaLaunchKernelEx(&cfg, ca_gather_kernel<256>, tin, tout, tq, inv, xchg, T, g, tqf, err);
      else
        e = cudaLaunchKernelEx(&cfg, ca_gather_kernel<128>, tin, tout, tq, inv, xchg, T, g, tqf, err);
    }
    if (e != cudaSuccess) return check_launch();
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
