// tc_cluster_dq.cu -- gradients of the orthogonal blocks, the permuted operand gathered in flight.
//
// Backward of the block-diagonal applies of "POET-X: Memory-efficient LLM
// Training by Scaling Orthogonal Transformation" (gist.science summary,
// sections 2.B-2.C and 2.E; the page leaves the backward to autograd, this is
// the plain chain rule).  For every block j
//     dQ_j[i][k] = sum_t G[t][j*b + i] * V[t][j*b + k]
// where exactly one operand is a permuted view of an activation:
//   R side  G = dy[:, perm_out] (gathered),  V = z                   (dQ_R)
//   P side  G = g_u,                         V = x[:, perm_in] (gathered)  (dQ_P)
// The permuted operand crosses HBM once, in its natural layout, and is
// gathered through the cluster exchange of tc_exchange.cuh (the same one the
// block applies use), so no permuted copy of it is ever written to HBM; the
// unpermuted operand's block columns come straight in by TMA.
//
// A cluster of C CTAs walks 64-token tiles (clusters take tiles
// round-robin); CTA c owns blocks [c*G, (c+1)*G).  The contraction runs over
// tokens on the tensor cores: tcgen05.mma with M = 128 rows i, N = b columns
// k, K = 16 tokens; the gathered part is K-major (feature rows of 64 tokens),
// the TMA tiles are MN-major (token rows of 64 features).  The fp32 sums stay
// in TMEM for the whole launch; at the end each CTA writes its blocks into the
// cluster's own slot of a partial-sum buffer [clusters][d/b][b][b] (clusters
// without tiles write zeros), which the consumer adds in slot order -- no
// atomics, so the result does not depend on scheduling.
//   warp 0      TMA: own natural columns of the permuted operand (exchange
//               input) and own blocks' columns of the other operand
//   warp 1      MMA (lane 0); lanes 1..C tell the writers a part was fetched
//   warps 2-9   movers: feature rows into the exchange ring
//   warps 10-13 epilogue: TMEM -> partial slot, 128-byte rows via shared memory
//   warp 14     loader: fetches this CTA's part of each exchange slot
//   warp 15     signals the readers when this CTA's rows of a slot are stored
#include "common.cuh"
#include "profile.cuh"
#include "tc.cuh"
#include "tc_exchange.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace poetx {
namespace tc {

namespace {

using namespace xchg;

constexpr int kDqThreads = 512;
constexpr int kSmemLimit = 232448;
constexpr int kPitch = 33;   // fp32 pitch of the 32 x 32 transpose tiles
constexpr int kOneCtaSmem = 120 * 1024;

struct DqGeo {
  int C, G, F;        // cluster size, blocks per CTA, natural features per CTA
  int NS, NR, NV;     // ring depths: own-column input, fetched parts, unpermuted operand
  int NX;             // exchange slots in the workspace ring
  int s_bytes;        // own-column input tile
  int r_bytes;        // fetched part (G*b feature rows of 128 bytes)
  int v_bytes;        // unpermuted operand tile (G*b columns x 64 tokens)
  int tmem_cols;
  int hdr, smem;
};

template <int B, bool GATHER_A>
__global__ void __launch_bounds__(kDqThreads, 1)
    cdq_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmV,
               const int32_t* __restrict__ inv, uint8_t* __restrict__ xring, float* __restrict__ part,
               int T, int nb, DqGeo g, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int halves = B / 128;
  const int C = g.C, G = g.G, F = g.F;
  const int s_off = g.hdr;
  const int r_off = s_off + g.NS * g.s_bytes;
  const int v_off = r_off + g.NR * g.r_bytes;
  const Bars br = bars_at(smem);
  uint32_t* table = reinterpret_cast<uint32_t*>(smem + kTableOff);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int c = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int n_clusters = gridDim.x / C;
  const int n_tiles = (T + TT - 1) / TT;
  const int n_it = cluster_iters(cluster_id, n_clusters, n_tiles);
  const size_t slot_stride = (size_t)C * g.r_bytes;
  uint8_t* ring = xring + (size_t)cluster_id * g.NX * slot_stride;

  if (threadIdx.x == 0) init_bars(br, C, kMovers, 1, kMovers);
  if (warp == 1) tmem_alloc(br.tmem_slot, (uint32_t)g.tmem_cols);
  gather_table<B>(table, inv, c, F, G);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // every CTA's barriers are initialised before any remote access
  tc_fence_after();
  const uint32_t tmem_base = *br.tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    // The two input streams advance independently: whichever ring has a free
    // stage gets its next tile (bounded: no progress for kWaitLimit polls is
    // recorded as a timeout).
    if (lane == 0) {
      int is = 0, iv = 0;
      uint32_t idle = 0;
      while (ok && (is < n_it || iv < n_it)) {
        bool moved_on = false;
        if (is < n_it && mbar_test_wait(br.s_empty + is % g.NS, ((is / g.NS) & 1) ^ 1)) {
          const int s = is % g.NS, tile = cluster_id + is * n_clusters;
          mbar_arrive_expect_tx(br.s_full + s, (uint32_t)g.s_bytes);
          uint8_t* sd = smem + s_off + s * g.s_bytes;
          for (int q = 0; q < F / 64; ++q)
            tma_load_2d(sd + q * (TT * 128), &tmP, c * F + q * 64, tile * TT, br.s_full + s);
          ++is;
          moved_on = true;
        }
        if (iv < n_it && mbar_test_wait(br.v_empty + iv % g.NV, ((iv / g.NV) & 1) ^ 1)) {
          const int v = iv % g.NV, tile = cluster_id + iv * n_clusters;
          mbar_arrive_expect_tx(br.v_full + v, (uint32_t)g.v_bytes);
          uint8_t* vd = smem + v_off + v * g.v_bytes;
          for (int jj = 0; jj < G; ++jj)
            for (int q = 0; q < B / 64; ++q)
              tma_load_2d(vd + jj * (B * TT * 2) + q * (TT * 128), &tmV, (c * G + jj) * B + q * 64,
                          tile * TT, br.v_full + v);
          ++iv;
          moved_on = true;
        }
        if (moved_on) {
          idle = 0;
        } else if (++idle > kWaitLimit) {
          raise_device_error(err, POETX_ERR_TIMEOUT);
          ok = false;
        }
      }
    }
  } else if (warp == 14) {
    // ---------------------------------------------------------------- loader
    if (lane == 0)
      loader_loop(br, g.NR, g.NX, g.r_bytes, smem + r_off, ring + (size_t)c * g.r_bytes, slot_stride,
                  n_it, ok, err);
  } else if (warp == 15) {
    // ---------------------------------------------------------------- signals to the readers
    signal_loop(br, g.NX, n_it, C, lane, ok, err);
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    const uint32_t idesc = idesc_bf16(128, B, !GATHER_A, GATHER_A);
    for (int it = 0; it < n_it && ok; ++it) {
      const int r = it % g.NR, v = it % g.NV;
      if (!(ok = mbar_wait(br.r_full + r, (it / g.NR) & 1, err))) break;
      if (lane >= 1) ack_fetch(br, it, g.NX, n_it, lane - 1, C);   // part fetched
      if (lane == 0) {
        if (!(ok = mbar_wait(br.v_full + v, (it / g.NV) & 1, err))) break;
        tc_fence_after();
        const uint32_t rb = smem_u32(smem + r_off + r * g.r_bytes);
        const uint32_t vb = smem_u32(smem + v_off + v * g.v_bytes);
        for (int jj = 0; jj < G; ++jj)
          for (int h = 0; h < halves; ++h) {
            const uint32_t d_tmem = tmem_base + (uint32_t)((jj * halves + h) * B);
#pragma unroll
            for (int kk = 0; kk < TT / 16; ++kk) {
              uint64_t adesc, bdesc;
              if (GATHER_A) {
                // A: gathered feature rows i (K-major); B: TMA tile, N = features k (MN-major)
                adesc = sw128_desc(rb + jj * (B * TT * 2) + h * (128 * 128) + kk * 32, 16, 1024);
                bdesc = sw128_desc(vb + jj * (B * TT * 2) + kk * 2048, TT * 128, 1024);
              } else {
                // A: TMA tile, M = features i (MN-major); B: gathered feature rows k (K-major)
                adesc = sw128_desc(vb + jj * (B * TT * 2) + h * 2 * (TT * 128) + kk * 2048, TT * 128, 1024);
                bdesc = sw128_desc(rb + jj * (B * TT * 2) + kk * 32, 16, 1024);
              }
              mma_bf16(d_tmem, adesc, bdesc, idesc, (it | kk) != 0 ? 1u : 0u);
            }
          }
        mma_commit(br.r_empty + r);
        mma_commit(br.v_empty + v);
      }
    }
    if (lane == 0 && ok && n_it > 0) mma_commit(br.q_full);   // every sum is final
  } else if (warp < 10) {
    // ---------------------------------------------------------------- movers
    const int pt = threadIdx.x - 64;
    for (int it = 0; it < n_it && ok; ++it) {
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
    // Lanes are rows i of the sums, registers 32 consecutive columns k; each
    // warp turns its 32 x 32 tiles through shared memory (the input ring is
    // idle once every product is done) so each store is a 128-byte row piece.
    const int quarter = warp % 4;
    const bool any = n_it > 0;
    if (any && mbar_wait(br.q_full, 0, err)) tc_fence_after();
    float* tt = reinterpret_cast<float*>(smem + s_off) + quarter * (32 * kPitch);
    float* slot = part + (size_t)cluster_id * nb * B * B;
    for (int jj = 0; jj < G; ++jj)
      for (int h = 0; h < halves; ++h) {
        float* dtile = slot + ((size_t)(c * G + jj) * B + h * 128 + quarter * 32) * B;
        for (int c0 = 0; c0 < B; c0 += 32) {
          uint32_t rr[32];
          if (any) {
            tmem_ld32(tmem_base + (uint32_t)((jj * halves + h) * B + c0) + ((uint32_t)(quarter * 32) << 16), rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = 0u;   // a cluster without tiles adds zero
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) tt[lane * kPitch + e] = __uint_as_float(rr[e]);
          __syncwarp();
#pragma unroll 8
          for (int q = 0; q < 32; ++q) dtile[(size_t)q * B + c0 + lane] = tt[q * kPitch + lane];
          __syncwarp();
        }
      }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves before its cluster is done with the exchange
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)g.tmem_cols);
  }
}

int pow2_cols(int used) {
  int c = 32;
  while (c < used) c *= 2;
  return c;
}

// Cluster sizes up to 8 (portable) only: where the blocks need more CTAs the
// permuted operand is gathered once into the scratch and summed by tc_dq
// (faster at the 2048 -> 5632 layer than 11-CTA clusters).
bool dq_geometry(int d, int b, DqGeo* out) {
  if ((b != 128 && b != 256) || d % b) return false;
  const int nb = d / b;
  const int halves = b / 128;
  const int order[7] = {8, 7, 6, 5, 4, 3, 2};
  for (int oi = 0; oi < 7; ++oi) {
    const int C = order[oi];
    if (nb % C) continue;
    DqGeo g;
    g.C = C;
    g.G = nb / C;
    g.F = d / C;
    if (g.F % 64 || g.G * halves * b > 512) continue;
    g.tmem_cols = pow2_cols(g.G * halves * b);
    g.s_bytes = TT * g.F * 2;
    g.r_bytes = g.G * b * TT * 2;
    g.v_bytes = g.G * b * TT * 2;
    g.hdr = (kTableOff + 4 * g.F + 1023) / 1024 * 1024;
    // (input, fetched, second operand) stages; a third second-operand stage
    // first (measured best at the square 2048 layer)
    const int cand[7][3] = {{2, 2, 3}, {3, 2, 2}, {2, 2, 2}, {2, 2, 1}, {2, 1, 1}, {1, 2, 1}, {1, 1, 1}};
    bool found = false;
    for (int ci = 0; ci < 7 && !found; ++ci) {
      const int smem = 1024 + g.hdr + cand[ci][0] * g.s_bytes + cand[ci][1] * g.r_bytes +
                       cand[ci][2] * g.v_bytes;
      // the epilogue's transpose tiles live in the input ring
      if (smem <= kSmemLimit && cand[ci][0] * g.s_bytes >= 4 * 32 * kPitch * 4) {
        g.NS = cand[ci][0];
        g.NR = cand[ci][1];
        g.NV = cand[ci][2];
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

const void* dq_kernel_ptr(int b, bool gather_a) {
  if (b == 256) return gather_a ? (const void*)cdq_kernel<256, true> : (const void*)cdq_kernel<256, false>;
  return gather_a ? (const void*)cdq_kernel<128, true> : (const void*)cdq_kernel<128, false>;
}

// Clusters of one launch over T tokens (as many as fit at once, at most one
// per tile; 0 if the kernel cannot be resident) and the exchange slots of each.
int dq_plan(int T, int b, DqGeo* g) {
  const void* kern = dq_kernel_ptr(b, true);
  if (set_max_dynamic_smem(dq_kernel_ptr(b, true), g->smem) != cudaSuccess ||
      set_max_dynamic_smem(dq_kernel_ptr(b, false), g->smem) != cudaSuccess ||
      (g->C > 8 && (cudaFuncSetAttribute(dq_kernel_ptr(b, true), cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
                    cudaFuncSetAttribute(dq_kernel_ptr(b, false), cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess))) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kDqThreads);
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
  if (n < 1) return 0;
  g->NX = ring_slots(n_tiles, n);
  return n;
}

}  // namespace

bool cluster_dq_supported(int d, int b) {
  DqGeo g;
  return dq_geometry(d, b, &g);
}

int cluster_dq_splits(int T, int d, int b) {
  DqGeo g;
  if (T <= 0 || !dq_geometry(d, b, &g)) return 0;
  return dq_plan(T, b, &g);
}

size_t cluster_dq_workspace_bytes(int T, int d, int b) {
  DqGeo g;
  if (T <= 0 || !dq_geometry(d, b, &g)) return 0;
  const int clusters = dq_plan(T, b, &g);
  return (size_t)clusters * g.NX * g.C * g.r_bytes;
}

poetx_status cluster_dq_bf16(const void* Pm, const void* Vc, const int32_t* inv, int T, int d, int b,
                             bool gather_a, float* part, void* ws, size_t ws_bytes, cudaStream_t s, int max_clusters) {
  DqGeo g;
  if (T <= 0 || !dq_geometry(d, b, &g)) return POETX_ERR_UNSUPPORTED;
  int clusters = dq_plan(T, b, &g);
  if (clusters < 1) return POETX_ERR_UNSUPPORTED;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  const int nb = d / b;
  if (!ws || ws_bytes < (size_t)clusters * g.NX * g.C * g.r_bytes || (reinterpret_cast<uintptr_t>(ws) & 255))
    return POETX_ERR_SHAPE;
  CUtensorMap tp, tv;
  if (!make_tmap_2d(&tp, Pm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, TT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tv, Vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)T, (uint64_t)d, TT, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return POETX_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * g.C);
  cfg.blockDim = dim3(kDqThreads);
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
  uint8_t* xr = static_cast<uint8_t*>(ws);
  {
    KernelScope ks_("tc_cluster_dq", s);
    cudaError_t e;
    if (b == 256)
      e = gather_a ? cudaLaunchKernelEx(&cfg, cdq_kernel<256, true>, tp, tv, inv, xr, part, T, nb, g, err)
                   : cudaLaunchKernelEx(&cfg, cdq_kernel<256, false>, tp, tv, inv, xr, part, T, nb, g, err);
    else
      e = gather_a ? cudaLaunchKernelEx(&cfg, cdq_kernel<128, true>, tp, tv, inv, xr, part, T, nb, g, err)
                   : cudaLaunchKernelEx(&cfg, cdq_kernel<128, false>, tp, tv, inv, xr, part, T, nb, g, err);
    if (e != cudaSuccess) return check_launch();
  }
  return check_launch();
}

}  // namespace tc
}  // namespace poetx
